"""Two forwards in flight at once, on two streams with a workspace each (the
library keeps no device state of its own between calls): their kernels share
the SMs — including the down GEMMs' per-window waits on their own gate/up
GEMMs — and every result equals the one of the same forward run alone, bit
for bit."""
import pytest

import moe_inputs
from gpu_util import need_gpu, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def test_concurrent_forwards_on_two_streams():
    torch = need_gpu()
    import combine_moe_route_04_gb300 as moe
    shapes = [(2048, 4096, 1536, 64, 8), (1024, 2048, 1024, 32, 4)]
    cases = []
    for i, shape in enumerate(shapes):
        T, H, I, E, k = shape
        s = moe.shape(*shape)
        d = dict(logits=to_dev(moe_inputs.make_logits(T, E, 51 + i)),
                 x=to_dev_bf16(moe_inputs.make_tokens(T, H, 51 + i)))
        d["wg"], d["wu"], d["wd"] = (to_dev_bf16(w) for w in moe_inputs.make_weights(E, H, I, 51 + i))
        ws = moe.alloc_workspace(s)
        out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
        moe.moe_forward(s, d["logits"], d["x"], d["wg"], d["wu"], d["wd"], out, ws)
        torch.cuda.synchronize()
        assert moe.last_device_status(ws) == 0
        cases.append((s, d, ws, out.clone()))

    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [torch.empty_like(c[3]) for c in cases]
    torch.cuda.synchronize()
    for _ in range(4):
        for (s, d, ws, _), out, st in zip(cases, outs, streams):
            with torch.cuda.stream(st):
                moe.moe_forward(s, d["logits"], d["x"], d["wg"], d["wu"], d["wd"], out, ws)
    torch.cuda.synchronize()
    for (s, d, ws, ref), out in zip(cases, outs):
        assert moe.last_device_status(ws) == 0
        assert torch.equal(out, ref)
