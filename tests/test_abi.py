"""CPU checks of the C ABI: the library builds and loads without a GPU, exports
every function include/moe.h declares, and its host-side validation rejects
bad shapes and pointers before launching anything."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def moe():
    from combine_moe_route_04_gb300 import _build
    _build.build()
    import combine_moe_route_04_gb300 as m
    m.load()
    return m


def _declared():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:moe_status|const char \*)\s*(moe_\w+)\s*\(", txt, re.M)))


def test_header_declares_the_abi():
    names = _declared()
    for n in ["moe_route", "moe_grouped_gemm_up", "moe_grouped_gemm_down", "moe_combine",
              "moe_forward"]:
        assert n in names


def test_library_exports_every_declared_symbol(moe):
    names = _declared()
    assert sorted(moe.EXPORTS) == names
    lib = moe.load()
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", moe.lib_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (moe_\w+)$", out, re.M))
    assert set(names) <= exported


def test_status_strings(moe):
    lib = moe.load()
    for code, name in moe.STATUS_NAMES.items():
        assert lib.moe_status_string(code).decode() == name


def test_capacity_matches_oracle(moe, oracle_mod):
    for (T, E, k) in [(1, 1, 1), (128, 8, 2), (64, 64, 8), (2048, 64, 8), (16384, 128, 8),
                      (3, 256, 16), (1000, 7, 3)]:
        mb, mr = moe.capacity(moe.shape(T, 128, 128, E, k))
        assert mb == oracle_mod.max_blocks(T, E, k)
        assert mr == 128 * mb


@pytest.mark.parametrize("bad", [(0, 256, 512, 8, 2), (128, 200, 512, 8, 2), (128, 256, 500, 8, 2),
                                 (128, 256, 512, 0, 1), (128, 256, 512, 8, 9), (128, 256, 512, 300, 2),
                                 (128, 256, 512, 32, 17), (128, 64, 512, 8, 2), (128, 256, 512, 8, 0)])
def test_unsupported_shapes_rejected(moe, bad):
    with pytest.raises(moe.MoEError) as ei:
        moe.workspace_size(moe.shape(*bad))
    assert ei.value.code == 2


def test_null_and_misaligned_pointers_rejected_before_launch(moe):
    lib = moe.load()
    s = moe.shape(128, 256, 512, 8, 2)
    P = ctypes.c_void_p
    good = 1 << 20             # never dereferenced: validation fails first
    rc = lib.moe_forward(ctypes.byref(s), None, good, good, good, good, good, good, None)
    assert rc == 1
    rc = lib.moe_forward(ctypes.byref(s), good + 4, good, good, good, good, good, good, None)
    assert rc == 3
    rc = lib.moe_combine(ctypes.byref(s), good, good, good, None, None, None)
    assert rc == 1
    rc = lib.moe_route(None, good, good, good, good, good, good, good, good, good, good, None)
    assert rc == 1


def test_workspace_size_covers_intermediates(moe):
    for cfg in [(128, 256, 512, 8, 2), (2048, 4096, 1536, 64, 8)]:
        s = moe.shape(*cfg)
        T, H, I, E, k = cfg
        mb, mr = moe.capacity(s)
        need = mr * H * 2 * 2 + mr * I * 2 + T * k * 12 + mr * 4
        assert moe.workspace_size(s) >= need


C_CLIENT = r"""
#include <stdio.h>
#include "moe.h"

int main(void) {
    moe_shape s = {2048, 4096, 1536, 64, 8};
    moe_shape bad = {2048, 4096, 1536, 64, 65};   /* k > E */
    int64_t mb = 0, mr = 0;
    size_t ws = 0;
    if (moe_capacity(&s, &mb, &mr) != MOE_OK) return 10;
    if (moe_workspace_size(&s, &ws) != MOE_OK) return 11;
    if (moe_workspace_size(&bad, &ws) != MOE_ERR_UNSUPPORTED_SHAPE) return 12;
    if (moe_workspace_size(&s, NULL) != MOE_ERR_INVALID_ARG) return 13;
    if (moe_workspace_size(&s, &ws) != MOE_OK) return 14;
    /* argument errors come back before anything touches a device */
    if (moe_forward(&s, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL) != MOE_ERR_INVALID_ARG) return 15;
    if (moe_forward(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL) != MOE_ERR_INVALID_ARG) return 16;
    printf("%lld %lld %zu %s\n", (long long)mb, (long long)mr, ws, moe_status_string(MOE_ERR_TIMEOUT));
    return 0;
}
"""


def test_header_and_library_serve_a_plain_c_client(moe, tmp_path):
    """include/moe.h compiles as strict C99 and a C program links the library
    and calls its host-side functions (no GPU needed for these)."""
    import shutil
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    libdir = os.path.dirname(moe.lib_path())
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe), "-L", libdir, "-l:" + os.path.basename(moe.lib_path()),
                    "-Wl,-rpath," + libdir], check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    mb, mr, ws, name = r.stdout.split()
    s = moe.shape(2048, 4096, 1536, 64, 8)
    assert (int(mb), int(mr)) == moe.capacity(s)
    assert int(ws) == moe.workspace_size(s)
    assert name == "MOE_ERR_TIMEOUT"
