"""Inside moe_forward the down GEMM does not wait for the whole gate/up grid:
each of its tiles waits until every gate/up tile of its token window has been
stored (a per-window count in the workspace).  If a tile read h too early, or
a count were left over from an earlier forward, its output would differ from
the one of the four step calls, which run each GEMM only after the previous
grid has completed.  So the forward must equal the step calls bit for bit:
  * on the pages-shaped workload (about two windows per expert);
  * on a skewed routing (one expert takes most rows: many down tiles wait on
    the same late windows);
  * on two shapes alternating on one workspace (counts cleared per forward)."""
import pytest

import moe_inputs
from gpu_util import need_gpu, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def _inputs(shape, seed, bias):
    T, H, I, E, k = shape
    logits = moe_inputs.make_logits(T, E, seed, bias=bias)
    x = moe_inputs.make_tokens(T, H, seed, row_signature=True)
    wg, wu, wd = moe_inputs.make_weights(E, H, I, seed)
    return {"logits": to_dev(logits), "x": to_dev_bf16(x), "wg": to_dev_bf16(wg), "wu": to_dev_bf16(wu),
            "wd": to_dev_bf16(wd)}


def _forward(moe, s, d, ws):
    import torch
    out = torch.empty((s.T, s.H), dtype=torch.bfloat16, device="cuda")
    moe.moe_forward(s, d["logits"], d["x"], d["wg"], d["wu"], d["wd"], out, ws)
    return out


def _steps(moe, s, d, ws):
    import torch
    r = moe.alloc_route_outputs(s)
    mb, mr = moe.capacity(s)
    moe.moe_route(s, d["logits"], r["topk_ids"], r["topk_w"], r["counts"], r["off_pad"], r["block_expert"],
                  r["num_blocks"], r["gather_idx"], r["scatter_idx"], ws)
    h = torch.empty((mr, s.I), dtype=torch.bfloat16, device="cuda")
    Y = torch.empty((mr, s.H), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((s.T, s.H), dtype=torch.bfloat16, device="cuda")
    moe.moe_grouped_gemm_up(s, d["x"], r["scatter_idx"], r["counts"], r["off_pad"], d["wg"], d["wu"], h, ws)
    moe.moe_grouped_gemm_down(s, h, r["counts"], r["off_pad"], d["wd"], Y, ws)
    moe.moe_combine(s, Y, r["scatter_idx"], r["topk_w"], out, ws)
    return out


@pytest.mark.parametrize("shape,bias", [((2048, 4096, 1536, 64, 8), "none"),
                                        ((4096, 1024, 768, 16, 4), "zipf3")])
def test_forward_equals_step_calls(shape, bias):
    torch = need_gpu()
    import combine_moe_route_04_gb300 as moe
    s = moe.shape(*shape)
    d = _inputs(shape, 71, bias)
    ws = moe.alloc_workspace(s)
    ref = _steps(moe, s, d, ws)
    assert moe.last_device_status(ws) == 0
    for _ in range(3):
        got = _forward(moe, s, d, ws)
        assert moe.last_device_status(ws) == 0
        assert torch.equal(got, ref)


def test_alternating_shapes_on_one_workspace():
    torch = need_gpu()
    import combine_moe_route_04_gb300 as moe
    shapes = [((1024, 1024, 768, 16, 4), "zipf3"), ((640, 512, 384, 8, 2), "none")]
    size = max(moe.workspace_size(moe.shape(*sh)) for sh, _ in shapes)
    ws = torch.zeros(size, dtype=torch.uint8, device="cuda")
    cases = []
    for sh, bias in shapes:
        s = moe.shape(*sh)
        d = _inputs(sh, 72, bias)
        cases.append((s, d, _steps(moe, s, d, ws)))
        assert moe.last_device_status(ws) == 0
    for _ in range(3):
        for s, d, ref in cases:
            got = _forward(moe, s, d, ws)
            assert moe.last_device_status(ws) == 0
            assert torch.equal(got, ref)


@pytest.mark.parametrize("shape,bias", [((2048, 4096, 1536, 64, 8), "none"),
                                        ((1024, 1024, 768, 16, 4), "zipf3")])
def test_back_to_back_forwards_keep_counters_clean(shape, bias):
    """Many forwards queued back to back on one stream, with no host
    synchronisation between them: each forward's tile counters and per-window
    counts must be back at zero before the next forward draws from them (a
    counter left dirty would skip or repeat tiles and report
    MOE_ERR_DEVICE_BOUNDS).  60 forwards in one burst, then 50 forwards each
    followed by a status check; every output equals the step calls'."""
    torch = need_gpu()
    import combine_moe_route_04_gb300 as moe
    s = moe.shape(*shape)
    d = _inputs(shape, 73, bias)
    ws = moe.alloc_workspace(s)
    ref = _steps(moe, s, d, ws)
    assert moe.last_device_status(ws) == 0
    outs = [torch.empty((s.T, s.H), dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    for i in range(60):
        o = outs[i % 4]
        moe.moe_forward(s, d["logits"], d["x"], d["wg"], d["wu"], d["wd"], o, ws)
    assert moe.last_device_status(ws) == 0
    for o in outs:
        assert torch.equal(o, ref)
    for i in range(50):
        got = _forward(moe, s, d, ws)
        assert moe.last_device_status(ws) == 0, "forward %d" % i
        assert torch.equal(got, ref), "forward %d" % i


def test_mixed_launch_regimes_queued_on_one_stream():
    """Forwards whose kernels let their dependents launch at different points,
    queued back to back on one stream with no host synchronisation, each
    layer on its own workspace.  The tiny layer's permutation lets the gate/up
    GEMM launch at entry (small gather) and its down GEMM loads weight slices
    before its window waits (one-wave gate/up GEMM); the decode and
    pages-shaped layers launch the gate/up GEMM after the permutation's wait;
    the fourth layer sits between.  Every output equals the step calls'."""
    torch = need_gpu()
    import combine_moe_route_04_gb300 as moe
    shapes = [((128, 256, 512, 8, 2), "none"), ((96, 2048, 512, 32, 4), "none"),
              ((64, 4096, 1536, 64, 8), "none"), ((2048, 4096, 1536, 64, 8), "none")]
    cases = []
    for i, (sh, bias) in enumerate(shapes):
        s = moe.shape(*sh)
        d = _inputs(sh, 74 + i, bias)
        ws = moe.alloc_workspace(s)
        ref = _steps(moe, s, d, ws)
        assert moe.last_device_status(ws) == 0
        outs = [torch.empty((s.T, s.H), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
        cases.append((s, d, ws, ref, outs))
    torch.cuda.synchronize()
    for r in range(12):
        for s, d, ws, _, outs in cases:
            moe.moe_forward(s, d["logits"], d["x"], d["wg"], d["wu"], d["wd"], outs[r % 2], ws)
    torch.cuda.synchronize()
    for s, d, ws, ref, outs in cases:
        assert moe.last_device_status(ws) == 0
        for o in outs:
            assert torch.equal(o, ref)
