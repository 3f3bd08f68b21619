"""The benchmark reports an ncu DRAM-traffic figure only while it was taken on
the current GEMM kernel code: the record carries a hash of the kernel source
with comments and blank lines left out.  A comment edit keeps the record
valid; a code edit voids it (the benchmark then reports null)."""
import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FILES = ("moe_gemm.cu", "moe_device.cuh")


def _copy_tree(tmp):
    dst = os.path.join(tmp, "combine_moe_route_04_gb300", "csrc")
    os.makedirs(dst)
    for n in FILES:
        shutil.copy(os.path.join(ROOT, "combine_moe_route_04_gb300", "csrc", n), dst)
    os.makedirs(os.path.join(tmp, "profiles"))
    shutil.copy(os.path.join(ROOT, "profiles", "dram_traffic.json"), os.path.join(tmp, "profiles"))
    return os.path.join(dst, "moe_gemm.cu")


def _hash_at(bench, root):
    saved = bench.ROOT
    bench.ROOT = root
    try:
        return bench.kernel_source_hash(), bench.recorded_traffic("grouped_gemm_window_kernel_up")
    finally:
        bench.ROOT = saved


def test_comment_edits_keep_the_record_and_code_edits_void_it(tmp_path):
    sys.path.insert(0, ROOT)
    import bench
    gemm = _copy_tree(str(tmp_path))
    h0, t0 = _hash_at(bench, str(tmp_path))
    assert h0 == bench.kernel_source_hash()

    with open(gemm, encoding="utf-8") as f:
        src = f.read()
    with open(gemm, "w", encoding="utf-8") as f:
        f.write("// an added comment line\n\n" + src.replace("namespace moe {", "namespace moe {  // trailing", 1))
    h1, t1 = _hash_at(bench, str(tmp_path))
    assert h1 == h0 and t1 == t0

    with open(gemm, "w", encoding="utf-8") as f:
        f.write(src.replace("constexpr int BK = 32;", "constexpr int BK = 64;", 1))
    h2, t2 = _hash_at(bench, str(tmp_path))
    assert h2 != h0 and t2 is None

