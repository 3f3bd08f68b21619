"""The gate/up GEMM's clusters draw their tiles from a counter kept in the
workspace (cleared by moe_workspace_init, cleared again by the last cluster of
every launch), and the routing's chunk CTAs count themselves in on another
(the CTA that arrives last scans the chunk histograms; the next kernel clears
it).  Checked on the GPU without faulting anything:
  * one workspace serves forwards of several shapes in turn, each exact;
  * a tile counter left at a value no launch can reach (what an uncleared
    workspace may hold) is reported as MOE_ERR_DEVICE_BOUNDS, the call
    returns, the counter is left cleared and the next forward is exact;
  * the same for the routing's chunk counter, through moe_forward and through
    the step call moe_route: no CTA scans, the call reports
    MOE_ERR_DEVICE_BOUNDS and routes every expert empty instead of using stale
    counts, the counter is cleared and the next call is exact."""
import numpy as np
import pytest

import moe_inputs
from gpu_util import assert_close_layer, host_u16, need_gpu, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

MOE_ERR_DEVICE_BOUNDS = 7
UP_TILE_COUNTER = 16        # int32 index in the workspace: its first 256 bytes hold the counters
ROUTE_COUNTER = 56

SHAPES = [  # (T, H, I, E, k, seed)
    (300, 512, 384, 5, 2, 91),
    (128, 256, 512, 8, 2, 92),
    (520, 256, 256, 16, 4, 93),
]


def _forward(moe, oracle_mod, shape, seed, ws):
    torch = need_gpu()
    T, H, I, E, k = shape
    logits = moe_inputs.make_logits(T, E, seed)
    x = moe_inputs.make_tokens(T, H, seed, row_signature=True)
    wg, wu, wd = moe_inputs.make_weights(E, H, I, seed)
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    moe.moe_forward(moe.shape(*shape), to_dev(logits), to_dev_bf16(x), to_dev_bf16(wg), to_dev_bf16(wu),
                    to_dev_bf16(wd), out, ws)
    return host_u16(out), (logits, x, wg, wu, wd, k)


def test_shapes_share_one_workspace(oracle_mod):
    torch = need_gpu()
    import combine_moe_route_04_gb300 as moe
    size = max(moe.workspace_size(moe.shape(*sh[:5])) for sh in SHAPES)
    ws = torch.zeros(size, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        for sh in SHAPES:
            got, args = _forward(moe, oracle_mod, sh[:5], sh[5], ws)
            assert moe.last_device_status(ws) == 0
            assert_close_layer(got, oracle_mod.layer(*args).out)
            assert int(ws.view(torch.int32)[UP_TILE_COUNTER]) == 0


def test_uncleared_tile_counter_is_reported_and_cleared(oracle_mod):
    """The gate/up GEMM stops drawing at once, so most windows are never
    stored.  On this shape the gate/up GEMM is one wave of tiles, so each
    down producer has claimed stages and loaded their weight slices before
    its window wait gives up: the forward must still report the bounds error
    (no wait left to run out its time limit, which would report a timeout),
    and the next forward must be exact."""
    torch = need_gpu()
    import combine_moe_route_04_gb300 as moe
    shape, seed = SHAPES[0][:5], SHAPES[0][5]
    ws = moe.alloc_workspace(moe.shape(*shape))
    ws.view(torch.int32)[UP_TILE_COUNTER] = 0x7FFFFFF0
    _forward(moe, oracle_mod, shape, seed, ws)
    assert moe.last_device_status(ws) == MOE_ERR_DEVICE_BOUNDS
    assert int(ws.view(torch.int32)[UP_TILE_COUNTER]) == 0
    got, args = _forward(moe, oracle_mod, shape, seed, ws)
    assert moe.last_device_status(ws) == 0
    assert_close_layer(got, oracle_mod.layer(*args).out)


def test_uncleared_route_counter_is_reported_and_cleared(oracle_mod):
    torch = need_gpu()
    import combine_moe_route_04_gb300 as moe
    shape, seed = SHAPES[2][:5], SHAPES[2][5]   # T = 520: 17 routing chunks
    s = moe.shape(*shape)
    ws = moe.alloc_workspace(s)
    # through moe_forward
    ws.view(torch.int32)[ROUTE_COUNTER] = 0x7FFFFFF0
    _forward(moe, oracle_mod, shape, seed, ws)
    assert moe.last_device_status(ws) == MOE_ERR_DEVICE_BOUNDS
    assert int(ws.view(torch.int32)[ROUTE_COUNTER]) == 0
    got, args = _forward(moe, oracle_mod, shape, seed, ws)
    assert moe.last_device_status(ws) == 0
    assert_close_layer(got, oracle_mod.layer(*args).out)
    # through the step call
    T, H, I, E, k = shape
    logits = moe_inputs.make_logits(T, E, seed)
    ref = oracle_mod.route(logits, k)
    r = moe.alloc_route_outputs(s)

    def route():
        moe.moe_route(s, to_dev(logits), r["topk_ids"], r["topk_w"], r["counts"], r["off_pad"], r["block_expert"],
                      r["num_blocks"], r["gather_idx"], r["scatter_idx"], ws)

    ws.view(torch.int32)[ROUTE_COUNTER] = 0x7FFFFFF0
    route()
    assert moe.last_device_status(ws) == MOE_ERR_DEVICE_BOUNDS
    assert int(ws.view(torch.int32)[ROUTE_COUNTER]) == 0
    assert int(r["num_blocks"].item()) == 0        # every expert routed empty, not stale counts
    assert int(r["counts"].abs().sum().item()) == 0
    route()
    assert moe.last_device_status(ws) == 0
    nb = int(r["num_blocks"].item())
    assert nb == ref.num_blocks
    assert np.array_equal(r["counts"].cpu().numpy(), ref.counts)
    assert np.array_equal(r["scatter_idx"].cpu().numpy(), ref.scatter_idx)
    assert np.array_equal(r["gather_idx"][:nb * 128].cpu().numpy(), ref.gather_idx)
