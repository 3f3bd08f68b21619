"""End-to-end GPU parity of moe_forward (the call the benchmark times):
  * the tiny workload and small edge shapes against the full oracle layer;
  * the four full-size workloads (T=2048..16384, H=4096, I=1536, E=64/128,
    k=8): routing, counts, block table and permutation bit-exact over the whole
    workload, and the WHOLE output, every real row of h and every real row of
    Y against the full oracle layer, element by element, with the relative
    Frobenius error taken over each whole tensor;
  * the same workloads' outputs of sampled tokens (first, last, random, and
    tokens whose rows sit at the ragged end of an expert group) against the
    oracle token by token, including their per-slot h and Y rows (the
    per-token path of the oracle, without its permutation);
  * determinism: two forwards give identical bits."""
import numpy as np
import pytest

import moe_inputs
from gpu_util import (assert_close_layer, assert_close_whole, assert_rows_close, host_u16, need_gpu, to_dev,
                      to_dev_bf16, ulp_dist_f32, W_ULPS)

pytestmark = pytest.mark.gpu


def _forward(moe, cfg_shape, inp, ws=None):
    torch = need_gpu()
    T, H, I, E, k = cfg_shape
    s = moe.shape(T, H, I, E, k)
    if ws is None:
        ws = moe.alloc_workspace(s)
    dev = {"logits": to_dev(inp["logits"]), "x": to_dev_bf16(inp["x"]),
           "wg": to_dev_bf16(inp["w_gate"]), "wu": to_dev_bf16(inp["w_up"]),
           "wd": to_dev_bf16(inp["w_down"])}
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    moe.moe_forward(s, dev["logits"], dev["x"], dev["wg"], dev["wu"], dev["wd"], out, ws)
    assert moe.last_device_status(ws) == 0
    return s, ws, dev, out


def _view_arrays(moe, s, ws):
    import torch
    v = moe.workspace_views(s, ws)
    mb, mr = moe.capacity(s)

    def grab(ptr, n, dtype):
        off = ptr - ws.data_ptr()
        nbytes = n * torch.empty(0, dtype=dtype).element_size()
        return ws[off:off + nbytes].view(dtype).cpu().numpy()

    T, k, E = s.T, s.k, s.E
    nb = int(grab(v.num_blocks, 1, torch.int32)[0])
    return {
        "num_blocks": nb,
        "topk_ids": grab(v.topk_ids, T * k, torch.int32).reshape(T, k),
        "topk_w": grab(v.topk_w, T * k, torch.float32).reshape(T, k),
        "counts": grab(v.counts, E, torch.int32),
        "off_pad": grab(v.off_pad, E + 1, torch.int32),
        "block_expert": grab(v.block_expert, mb, torch.int32)[:nb],
        "gather_idx": grab(v.gather_idx, mr, torch.int32)[:nb * 128],
        "scatter_idx": grab(v.scatter_idx, T * k, torch.int32).reshape(T, k),
        "h_ptr": v.h, "Y_ptr": v.Y, "Xp_ptr": v.Xp,
    }


def _rows_of(ws, ptr, rows, width):
    import torch
    off = ptr - ws.data_ptr()
    buf = ws[off:off + (int(rows.max()) + 1) * width * 2].view(torch.int16).view(-1, width)
    idx = torch.from_numpy(np.asarray(rows, np.int64)).cuda()
    return buf[idx].cpu().numpy().view(np.uint16)


SMALL = {
    "tiny_cfg": (moe_inputs.config(1).shape, 1001),
    "multi_tile": ((300, 512, 384, 5, 2), 77),
    "h_tail_128": ((200, 384, 256, 3, 2), 78),
    "single_token": ((1, 256, 256, 8, 2), 79),
    "k_equals_E": ((70, 256, 128, 4, 4), 80),
    "many_experts": ((96, 256, 128, 256, 16), 81),
    "smallest_dims": ((50, 128, 128, 3, 2), 82),      # H = I = 128: the down tile is half outside, K = 4 stages
    "widest_hidden": ((8, 32768, 128, 2, 1), 83),     # H at its limit: 1024 K stages up, 64 down tiles per window
    "widest_inner": ((40, 128, 32768, 3, 2), 84),     # I at its limit: 128 up tiles per window, 1024 K stages down
}


@pytest.mark.parametrize("name", list(SMALL))
def test_forward_small_full_oracle(oracle_mod, name):
    import combine_moe_route_04_gb300 as moe
    (T, H, I, E, k), seed = SMALL[name]
    inp = {"logits": moe_inputs.make_logits(T, E, seed),
           "x": moe_inputs.make_tokens(T, H, seed, row_signature=True)}
    inp["w_gate"], inp["w_up"], inp["w_down"] = moe_inputs.make_weights(E, H, I, seed)
    s, ws, dev, out = _forward(moe, (T, H, I, E, k), inp)
    ref = oracle_mod.layer(inp["logits"], inp["x"], inp["w_gate"], inp["w_up"], inp["w_down"], k)
    assert_rows_close(host_u16(out), ref.out, "out")
    v = _view_arrays(moe, s, ws)
    assert v["num_blocks"] == ref.route.num_blocks
    assert np.array_equal(v["topk_ids"], ref.route.topk_ids)
    assert np.array_equal(v["gather_idx"], ref.route.gather_idx)
    assert np.array_equal(v["scatter_idx"], ref.route.scatter_idx)
    # the gathered rows the up GEMM read: Xp[r] = X[gather_idx[r]], bit for bit
    real = np.nonzero(ref.route.gather_idx >= 0)[0]
    xp = _rows_of(ws, v["Xp_ptr"], real, H)
    assert np.array_equal(xp, inp["x"][ref.route.gather_idx[real]])


def _sample_tokens(ref_route, T, rng, n_random=29):
    toks = {0, 1, T - 1}
    toks.update(int(t) for t in rng.choice(T, size=min(n_random, T), replace=False))
    # tokens owning the last real row of a few expert groups (padding-adjacent rows)
    r = ref_route
    nonempty = np.nonzero(r.counts > 0)[0]
    for e in rng.choice(nonempty, size=min(8, nonempty.size), replace=False):
        last_row = r.off_pad[e] + r.counts[e] - 1
        toks.add(int(r.gather_idx[last_row]))
    return np.array(sorted(toks), dtype=np.int32)


@pytest.mark.slow
@pytest.mark.parametrize("n", [2, 3, 4, 5])
def test_forward_full_workload_sampled(oracle_mod, n):
    import combine_moe_route_04_gb300 as moe
    cfg = moe_inputs.config(n)
    inp = moe_inputs.make_inputs(cfg)
    s, ws, dev, out = _forward(moe, cfg.shape, inp)
    ref_route = oracle_mod.route(inp["logits"], cfg.k)
    v = _view_arrays(moe, s, ws)
    # routing over the whole workload: bit-exact
    assert v["num_blocks"] == ref_route.num_blocks
    assert np.array_equal(v["topk_ids"], ref_route.topk_ids)
    assert np.array_equal(v["counts"], ref_route.counts)
    assert np.array_equal(v["off_pad"], ref_route.off_pad)
    assert np.array_equal(v["block_expert"], ref_route.block_expert)
    assert np.array_equal(v["gather_idx"], ref_route.gather_idx)
    assert np.array_equal(v["scatter_idx"], ref_route.scatter_idx)
    assert ulp_dist_f32(v["topk_w"], ref_route.topk_w).max() <= W_ULPS
    # sampled tokens, one by one
    rng = np.random.default_rng(100 + n)
    toks = _sample_tokens(ref_route, cfg.T, rng)
    o_ref, h_ref, y_ref = oracle_mod.tokens_out(toks, ref_route.topk_ids, ref_route.topk_w,
                                                inp["x"], inp["w_gate"], inp["w_up"], inp["w_down"],
                                                want_rows=True)
    rows = ref_route.scatter_idx[toks].ravel()
    h_got = _rows_of(ws, v["h_ptr"], rows, cfg.I)
    y_got = _rows_of(ws, v["Y_ptr"], rows, cfg.H)
    assert_rows_close(h_got, h_ref.reshape(-1, cfg.I), "h rows")
    assert_rows_close(y_got, y_ref.reshape(-1, cfg.H), "Y rows")
    o_got = host_u16(out)[toks]
    assert_rows_close(o_got, o_ref, "out (sampled tokens)")
    # every output finite
    import torch
    assert bool(torch.isfinite(out.float()).all())


@pytest.mark.slow
def test_forward_maximum_token_count(oracle_mod):
    """moe_forward at the largest T the shape check accepts (2^22 tokens, with
    the smallest H and I): 8.4 M permuted rows, 32 776 token windows, and the
    gather and combine striding over 4 M tokens.  Routing bit-exact over every
    token; sampled tokens' h, Y and out rows against the oracle."""
    import combine_moe_route_04_gb300 as moe
    T, H, I, E, k = 1 << 22, 128, 128, 8, 2
    seed = 85
    inp = {"logits": moe_inputs.make_logits(T, E, seed), "x": moe_inputs.make_tokens(T, H, seed)}
    inp["w_gate"], inp["w_up"], inp["w_down"] = moe_inputs.make_weights(E, H, I, seed)
    s, ws, dev, out = _forward(moe, (T, H, I, E, k), inp)
    ref_route = oracle_mod.route(inp["logits"], k)
    v = _view_arrays(moe, s, ws)
    assert v["num_blocks"] == ref_route.num_blocks
    assert np.array_equal(v["topk_ids"], ref_route.topk_ids)
    assert np.array_equal(v["counts"], ref_route.counts)
    assert np.array_equal(v["off_pad"], ref_route.off_pad)
    assert np.array_equal(v["gather_idx"], ref_route.gather_idx)
    assert np.array_equal(v["scatter_idx"], ref_route.scatter_idx)
    assert ulp_dist_f32(v["topk_w"], ref_route.topk_w).max() <= W_ULPS
    rng = np.random.default_rng(185)
    toks = _sample_tokens(ref_route, T, rng)
    o_ref, h_ref, y_ref = oracle_mod.tokens_out(toks, ref_route.topk_ids, ref_route.topk_w,
                                                inp["x"], inp["w_gate"], inp["w_up"], inp["w_down"],
                                                want_rows=True)
    rows = ref_route.scatter_idx[toks].ravel()
    assert_rows_close(_rows_of(ws, v["h_ptr"], rows, I), h_ref.reshape(-1, I), "h rows")
    assert_rows_close(_rows_of(ws, v["Y_ptr"], rows, H), y_ref.reshape(-1, H), "Y rows")
    assert_rows_close(host_u16(out)[toks], o_ref, "out (sampled tokens)")
    import torch
    assert bool(torch.isfinite(out.float()).all())


def _whole_rows(ws, ptr, nrows, width):
    import torch
    off = ptr - ws.data_ptr()
    return ws[off:off + nrows * width * 2].view(torch.int16).cpu().numpy().view(np.uint16).reshape(nrows, width)


@pytest.mark.slow
@pytest.mark.parametrize("n", [3, 2, 4, 5])
def test_forward_full_workload_whole_output(oracle_mod, n):
    """moe_forward on the full-size workload against the full oracle layer:
    routing bit-exact, then the whole out [T, H], every real row of h and of Y,
    each within the layer tolerance element by element and by relative
    Frobenius error over the whole tensor."""
    import combine_moe_route_04_gb300 as moe
    cfg = moe_inputs.config(n)
    inp = moe_inputs.make_inputs(cfg)
    s, ws, dev, out = _forward(moe, cfg.shape, inp)
    ref = oracle_mod.layer(inp["logits"], inp["x"], inp["w_gate"], inp["w_up"], inp["w_down"], cfg.k)
    v = _view_arrays(moe, s, ws)
    assert v["num_blocks"] == ref.route.num_blocks
    assert np.array_equal(v["topk_ids"], ref.route.topk_ids)
    assert np.array_equal(v["counts"], ref.route.counts)
    assert np.array_equal(v["off_pad"], ref.route.off_pad)
    assert np.array_equal(v["block_expert"], ref.route.block_expert)
    assert np.array_equal(v["gather_idx"], ref.route.gather_idx)
    assert np.array_equal(v["scatter_idx"], ref.route.scatter_idx)
    assert ulp_dist_f32(v["topk_w"], ref.route.topk_w).max() <= W_ULPS
    real = np.nonzero(ref.route.gather_idx >= 0)[0]
    assert real.size == cfg.T * cfg.k
    rows = ref.route.num_blocks * 128
    h_got = _whole_rows(ws, v["h_ptr"], rows, cfg.I)[real]
    assert_close_whole(h_got, ref.h[real], "h (every real row)")
    del h_got
    y_got = _whole_rows(ws, v["Y_ptr"], rows, cfg.H)[real]
    assert_close_whole(y_got, ref.Y[real], "Y (every real row)")
    del y_got
    err, fro = assert_close_whole(host_u16(out), ref.out, "out (whole output)")
    print("workload %d whole output: max |err| %.4g, relative Frobenius %.3g" % (n, err, fro))


def test_forward_deterministic_and_reusable_workspace(oracle_mod):
    import combine_moe_route_04_gb300 as moe
    (T, H, I, E, k), seed = SMALL["multi_tile"]
    inp = {"logits": moe_inputs.make_logits(T, E, seed), "x": moe_inputs.make_tokens(T, H, seed)}
    inp["w_gate"], inp["w_up"], inp["w_down"] = moe_inputs.make_weights(E, H, I, seed)
    s, ws, dev, out1 = _forward(moe, (T, H, I, E, k), inp)
    a = host_u16(out1)
    s, ws, dev, out2 = _forward(moe, (T, H, I, E, k), inp, ws=ws)
    assert np.array_equal(a, host_u16(out2))
