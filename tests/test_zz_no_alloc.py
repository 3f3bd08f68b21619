"""moe_route_noalloc: the routing entry point for callers that may not
allocate device memory (a plugin whose host framework owns all device memory
and passes it only inputs and outputs, or a deployment that forbids
allocation once it is running).  Its scratch is a fixed array inside the
library, so these tests check, through the C ABI, that two calls in a row give
exactly what moe_route gives with a caller workspace, and that a shape needing
more scratch than the fixed array is refused before anything runs.

This file is named to be collected last, so a stop-at-first-failure run has
already run every other test; it also passes on its own in a fresh process."""
import ctypes

import numpy as np
import pytest

import moe_inputs
from gpu_util import W_ULPS, need_gpu, to_dev, ulp_dist_f32


def _route_with_workspace(moe, s, logits_dev):
    bufs = moe.alloc_route_outputs(s)
    ws = moe.alloc_workspace(s)
    moe.moe_route(s, logits_dev, bufs["topk_ids"], bufs["topk_w"], bufs["counts"], bufs["off_pad"],
                  bufs["block_expert"], bufs["num_blocks"], bufs["gather_idx"], bufs["scatter_idx"], ws)
    assert moe.last_device_status(ws) == 0
    return bufs


def _route_noalloc_c_abi(moe, s, logits_dev, bufs, stream):
    lib = moe.load()
    rc = lib.moe_route_noalloc(ctypes.byref(s), logits_dev.data_ptr(), bufs["topk_ids"].data_ptr(),
                               bufs["topk_w"].data_ptr(), bufs["counts"].data_ptr(),
                               bufs["off_pad"].data_ptr(), bufs["block_expert"].data_ptr(),
                               bufs["num_blocks"].data_ptr(), bufs["gather_idx"].data_ptr(),
                               bufs["scatter_idx"].data_ptr(), stream)
    return rc


def _compare(a, b):
    nb = int(a["num_blocks"].item())
    assert nb == int(b["num_blocks"].item())
    for key in ("topk_ids", "counts", "off_pad", "scatter_idx"):
        assert np.array_equal(a[key].cpu().numpy(), b[key].cpu().numpy()), key
    assert np.array_equal(a["block_expert"][:nb].cpu().numpy(), b["block_expert"][:nb].cpu().numpy())
    assert np.array_equal(a["gather_idx"][:nb * 128].cpu().numpy(), b["gather_idx"][:nb * 128].cpu().numpy())
    # same kernels, same arithmetic: the weights agree to the bit, well inside
    # the routing tolerance used elsewhere
    assert ulp_dist_f32(a["topk_w"].cpu().numpy(), b["topk_w"].cpu().numpy()).max() <= W_ULPS


@pytest.mark.gpu
def test_noalloc_route_matches_workspace_route_on_two_calls():
    torch = need_gpu()
    import combine_moe_route_04_gb300 as moe
    stream = torch.cuda.current_stream().cuda_stream
    # two different inputs in a row: the second call must not see the first's scratch
    for n in (5, 4):
        cfg = moe_inputs.config(n)
        logits = to_dev(moe_inputs.make_logits(cfg.T, cfg.E, cfg.seed, cfg.logit_bias))
        s = moe.shape(*cfg.shape)
        ref = _route_with_workspace(moe, s, logits)
        got = moe.alloc_route_outputs(s)
        rc = _route_noalloc_c_abi(moe, s, logits, got, stream)
        assert rc == 0, moe.STATUS_NAMES.get(rc, rc)
        torch.cuda.synchronize()
        _compare(got, ref)


@pytest.mark.gpu
def test_noalloc_route_refuses_shapes_beyond_its_scratch():
    torch = need_gpu()
    import combine_moe_route_04_gb300 as moe
    # E * ceil(T/32) = 256 * 1025 > 262144 entries of fixed scratch
    s = moe.shape(32800, 128, 128, 256, 8)
    bufs = {k: torch.empty(1, dtype=torch.int32, device="cuda") for k in
            ("topk_ids", "topk_w", "counts", "off_pad", "block_expert", "num_blocks", "gather_idx",
             "scatter_idx")}
    logits = torch.empty(1, dtype=torch.float32, device="cuda")
    rc = _route_noalloc_c_abi(moe, s, logits, bufs, torch.cuda.current_stream().cuda_stream)
    assert moe.STATUS_NAMES[rc] == "MOE_ERR_SCRATCH_LIMIT"
