"""A bounded wait that runs out, on the GPU, without faulting it: the
diagnostic kernel waits on an mbarrier that nothing arrives on, through the
same bounded wait as the GEMM and combine pipelines.  After the limit (2 s of
%globaltimer) it records a timeout in the workspace status word and returns.
The host reads MOE_ERR_TIMEOUT, the word is cleared, and the same context then
runs a whole layer exactly."""
import time

import pytest

import moe_inputs
from gpu_util import assert_close_layer, host_u16, need_gpu, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

MOE_ERR_TIMEOUT = 6
WAIT_LIMIT_S = 2.0


def test_wait_that_runs_out_is_reported_and_context_stays_usable(oracle_mod):
    torch = need_gpu()
    import combine_moe_route_04_gb300 as moe
    shape = (300, 512, 384, 5, 2)
    s = moe.shape(*shape)
    ws = moe.alloc_workspace(s)
    torch.cuda.synchronize()

    t0 = time.perf_counter()
    moe.check_wait_timeout(ws)
    status = moe.last_device_status(ws)          # synchronises
    elapsed = time.perf_counter() - t0
    assert status == MOE_ERR_TIMEOUT
    assert WAIT_LIMIT_S <= elapsed < 10 * WAIT_LIMIT_S
    assert moe.last_device_status(ws) == 0       # read once, then cleared

    T, H, I, E, k = shape
    logits = moe_inputs.make_logits(T, E, 97)
    x = moe_inputs.make_tokens(T, H, 97, row_signature=True)
    wg, wu, wd = moe_inputs.make_weights(E, H, I, 97)
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    moe.moe_forward(s, to_dev(logits), to_dev_bf16(x), to_dev_bf16(wg), to_dev_bf16(wu), to_dev_bf16(wd), out, ws)
    assert moe.last_device_status(ws) == 0
    assert_close_layer(host_u16(out), oracle_mod.layer(logits, x, wg, wu, wd, k).out)


def test_wait_check_rejects_bad_workspace():
    need_gpu()
    import combine_moe_route_04_gb300 as moe
    with pytest.raises(moe.MoEError):
        moe.check_wait_timeout(None)


def test_unread_earlier_error_does_not_stop_a_forward(oracle_mod):
    """The down GEMM's per-window waits give up only on an error raised during
    the current forward: an earlier error nobody has read yet (here the
    diagnostic's timeout) leaves the next forward exact, and is still the one
    moe_last_device_status reports."""
    torch = need_gpu()
    import combine_moe_route_04_gb300 as moe
    shape = (520, 256, 256, 16, 4)
    s = moe.shape(*shape)
    ws = moe.alloc_workspace(s)
    moe.check_wait_timeout(ws)                   # sets the timeout bit; not read here
    T, H, I, E, k = shape
    logits = moe_inputs.make_logits(T, E, 98)
    x = moe_inputs.make_tokens(T, H, 98)
    wg, wu, wd = moe_inputs.make_weights(E, H, I, 98)
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    moe.moe_forward(s, to_dev(logits), to_dev_bf16(x), to_dev_bf16(wg), to_dev_bf16(wu), to_dev_bf16(wd), out, ws)
    assert moe.last_device_status(ws) == MOE_ERR_TIMEOUT
    assert_close_layer(host_u16(out), oracle_mod.layer(logits, x, wg, wu, wd, k).out)
    assert moe.last_device_status(ws) == 0
