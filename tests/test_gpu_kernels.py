"""Per-kernel GPU parity: the grouped gate/up GEMM (with its row gather, and
on rows already in expert order), the grouped down GEMM and the combine, each
fed the oracle's own inputs (its route and, for down and combine, its h / Y),
so an error is localised to one kernel.  Shapes span
several row blocks and column tiles, ragged expert groups, an expert of
exactly 128 and one of 129 rows, and empty experts."""
import numpy as np
import pytest

import moe_inputs
from gpu_util import (assert_rows_close, host_u16, need_gpu, to_dev, to_dev_bf16)

pytestmark = pytest.mark.gpu

CASES = {
    # name: (T, H, I, E, k, seed, special)
    "tiny_cfg": (128, 256, 512, 8, 2, 1001, None),
    "multi_tile": (300, 512, 384, 5, 2, 77, None),
    "h_tail_128": (200, 384, 256, 3, 2, 78, None),       # H % 256 == 128: half-outside down tile
    "boundaries": (258, 256, 256, 4, 1, 79, "boundaries"),
    "one_expert": (257, 256, 128, 1, 1, 80, None),
    "wide_k": (40, 256, 256, 16, 16, 81, None),
}


def make_case(name):
    T, H, I, E, k, seed, special = CASES[name]
    logits = moe_inputs.make_logits(T, E, seed)
    if special == "boundaries":
        logits = np.full((T, E), -10.0, dtype=np.float32)
        logits[:128, 0] = 10
        logits[128:257, 1] = 10
        logits[257, 3] = 10
    x = moe_inputs.make_tokens(T, H, seed, row_signature=True)
    wg, wu, wd = moe_inputs.make_weights(E, H, I, seed)
    return (T, H, I, E, k), logits, x, wg, wu, wd


def upload_route(moe, s, r):
    torch = need_gpu()
    mb, mr = moe.capacity(s)
    be = np.zeros(mb, np.int32)
    be[:r.num_blocks] = r.block_expert
    g = np.full(mr, -1, np.int32)
    g[:r.num_blocks * 128] = r.gather_idx
    return {"off_pad": to_dev(r.off_pad), "block_expert": to_dev(be), "counts": to_dev(r.counts),
            "num_blocks": to_dev(np.array([r.num_blocks], np.int32)), "gather_idx": to_dev(g),
            "scatter_idx": to_dev(r.scatter_idx), "topk_w": to_dev(r.topk_w)}


@pytest.mark.parametrize("name", list(CASES))
def test_grouped_gemms_and_combine(oracle_mod, name):
    torch = need_gpu()
    import combine_moe_route_04_gb300 as moe
    (T, H, I, E, k), logits, x, wg, wu, wd = make_case(name)
    ref = oracle_mod.layer(logits, x, wg, wu, wd, k)
    r = ref.route
    s = moe.shape(T, H, I, E, k)
    mb, mr = moe.capacity(s)
    d = upload_route(moe, s, r)
    ws = moe.alloc_workspace(s)
    real = np.nonzero(r.gather_idx >= 0)[0]

    # up GEMM on the oracle's route
    h = torch.empty((mr, I), dtype=torch.bfloat16, device="cuda")
    moe.moe_grouped_gemm_up(s, to_dev_bf16(x), d["scatter_idx"], d["counts"], d["off_pad"],
                            to_dev_bf16(wg), to_dev_bf16(wu), h, ws)
    assert moe.last_device_status(ws) == 0
    h_got = host_u16(h)[:r.num_blocks * 128]
    assert_rows_close(h_got[real], ref.h[real], "h")

    # the same GEMM on rows already in expert order (no gather): Xp[r] = X[gather_idx[r]]
    xp = np.zeros((mr, H), np.uint16)
    xp[real] = x[r.gather_idx[real]]
    h2 = torch.empty((mr, I), dtype=torch.bfloat16, device="cuda")
    moe.moe_grouped_gemm_up_rows(s, to_dev_bf16(xp), d["counts"], d["off_pad"], to_dev_bf16(wg),
                                 to_dev_bf16(wu), h2, ws)
    assert moe.last_device_status(ws) == 0
    assert np.array_equal(host_u16(h2)[real], h_got[real])

    # down GEMM on the oracle's h
    h_ref_dev = torch.zeros((mr, I), dtype=torch.bfloat16, device="cuda")
    h_ref_dev[:r.num_blocks * 128] = to_dev_bf16(ref.h)
    Y = torch.empty((mr, H), dtype=torch.bfloat16, device="cuda")
    moe.moe_grouped_gemm_down(s, h_ref_dev, d["counts"], d["off_pad"], to_dev_bf16(wd), Y, ws)
    assert moe.last_device_status(ws) == 0
    y_got = host_u16(Y)[:r.num_blocks * 128]
    assert_rows_close(y_got[real], ref.Y[real], "Y")

    # combine on the oracle's Y: same float32 arithmetic in the same order -> bit-exact
    Y_ref_dev = torch.zeros((mr, H), dtype=torch.bfloat16, device="cuda")
    Y_ref_dev[:r.num_blocks * 128] = to_dev_bf16(ref.Y)
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    moe.moe_combine(s, Y_ref_dev, d["scatter_idx"], d["topk_w"], out, ws)
    assert moe.last_device_status(ws) == 0
    assert np.array_equal(host_u16(out), ref.out)


def test_gemm_up_bitwise_deterministic(oracle_mod):
    torch = need_gpu()
    import combine_moe_route_04_gb300 as moe
    (T, H, I, E, k), logits, x, wg, wu, wd = make_case("multi_tile")
    r = oracle_mod.route(logits, k)
    s = moe.shape(T, H, I, E, k)
    mb, mr = moe.capacity(s)
    d = upload_route(moe, s, r)
    ws = moe.alloc_workspace(s)
    outs = []
    for _ in range(2):
        h = torch.zeros((mr, I), dtype=torch.bfloat16, device="cuda")
        moe.moe_grouped_gemm_up(s, to_dev_bf16(x), d["scatter_idx"], d["counts"], d["off_pad"],
                                to_dev_bf16(wg), to_dev_bf16(wu), h, ws)
        outs.append(host_u16(h)[:r.num_blocks * 128][r.gather_idx >= 0])
    assert np.array_equal(outs[0], outs[1])
