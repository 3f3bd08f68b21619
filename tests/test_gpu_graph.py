"""CUDA graphs: moe_forward, and the four step calls, recorded by stream
capture (the kernel launches with their programmatic-dependent-launch edges)
and replayed.  Every replay equals the same calls made directly, bit for
bit, also when new inputs are copied into the captured buffers between
replays; the pages-shaped workload's per-window hand-off between the GEMMs
runs inside the graph too."""
import numpy as np
import pytest

import moe_inputs
from gpu_util import need_gpu, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape", [(128, 256, 512, 8, 2), (2048, 4096, 1536, 64, 8)])
def test_graph_replay_equals_direct_calls(shape):
    torch = need_gpu()
    import combine_moe_route_04_gb300 as moe
    T, H, I, E, k = shape
    s = moe.shape(*shape)
    wg, wu, wd = (to_dev_bf16(w) for w in moe_inputs.make_weights(E, H, I, 41))
    inputs = [(to_dev(moe_inputs.make_logits(T, E, seed)), to_dev_bf16(moe_inputs.make_tokens(T, H, seed)))
              for seed in (42, 43, 44)]
    logits = torch.empty_like(inputs[0][0])
    x = torch.empty_like(inputs[0][1])
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    ws = moe.alloc_workspace(s)

    refs = []
    for lg, xx in inputs:
        logits.copy_(lg)
        x.copy_(xx)
        moe.moe_forward(s, logits, x, wg, wu, wd, out, ws)
        refs.append(out.clone())
    assert moe.last_device_status(ws) == 0
    assert not torch.equal(refs[0], refs[1])

    g = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            moe.moe_forward(s, logits, x, wg, wu, wd, out, ws)
    torch.cuda.synchronize()
    for _ in range(2):
        for (lg, xx), ref in zip(inputs, refs):
            logits.copy_(lg)
            x.copy_(xx)
            out.zero_()
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(out, ref)
    assert moe.last_device_status(ws) == 0


def test_step_calls_captured_in_one_graph():
    """The four step calls recorded into one graph (route -> up -> down ->
    combine, each on buffers of the caller) replay to the same bits as the
    same calls made directly."""
    torch = need_gpu()
    import combine_moe_route_04_gb300 as moe
    shape = (520, 512, 384, 16, 4)
    T, H, I, E, k = shape
    s = moe.shape(*shape)
    logits = to_dev(moe_inputs.make_logits(T, E, 45))
    x = to_dev_bf16(moe_inputs.make_tokens(T, H, 45))
    wg, wu, wd = (to_dev_bf16(w) for w in moe_inputs.make_weights(E, H, I, 45))
    ws = moe.alloc_workspace(s)
    r = moe.alloc_route_outputs(s)
    mb, mr = moe.capacity(s)
    h = torch.empty((mr, I), dtype=torch.bfloat16, device="cuda")
    Y = torch.empty((mr, H), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")

    def steps():
        moe.moe_route(s, logits, r["topk_ids"], r["topk_w"], r["counts"], r["off_pad"], r["block_expert"],
                      r["num_blocks"], r["gather_idx"], r["scatter_idx"], ws)
        moe.moe_grouped_gemm_up(s, x, r["scatter_idx"], r["counts"], r["off_pad"], wg, wu, h, ws)
        moe.moe_grouped_gemm_down(s, h, r["counts"], r["off_pad"], wd, Y, ws)
        moe.moe_combine(s, Y, r["scatter_idx"], r["topk_w"], out, ws)

    steps()
    torch.cuda.synchronize()
    ref = out.clone()
    assert moe.last_device_status(ws) == 0
    g = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            steps()
    torch.cuda.synchronize()
    for _ in range(3):
        out.zero_()
        h.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    assert moe.last_device_status(ws) == 0
