"""Pins of the oracle's expert FFN, grouped path and combine against closed
forms (one-hot inputs), library routines (torch float64 matmul, scipy's
logistic), special cases of the layer (k=1 & E=1 dense SwiGLU, identical
experts, k=E mixture, scaling of W_down by 2) and a dense brute-force form that
evaluates every expert on every token without any permutation."""
import numpy as np
import pytest
import torch
from scipy.special import expit

import moe_inputs


def _bf16_bits_t(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _f(bits):
    return torch.from_numpy((np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32))


def _ulp_diff(a, b):
    """Distance in bf16 ulps between two bf16 bit arrays (same sign assumed
    for non-zero pairs; zero-crossings count as large)."""
    a = np.asarray(a, np.int32)
    b = np.asarray(b, np.int32)
    sa = np.where(a & 0x8000, -(a & 0x7FFF), a & 0x7FFF)
    sb = np.where(b & 0x8000, -(b & 0x7FFF), b & 0x7FFF)
    return np.abs(sa - sb)


def _small_layer(T, H, I, E, k, seed):
    logits = moe_inputs.make_logits(T, E, seed)
    x = moe_inputs.make_tokens(T, H, seed)
    wg, wu, wd = moe_inputs.make_weights(E, H, I, seed, threads=1)
    return logits, x, wg, wu, wd


def _dense_reference(logits, x, wg, wu, wd, ids, w):
    """Every expert on every token in torch float64, with the layer's rounding
    points (g,u -> f32; silu(g)*u -> f32 -> bf16; y -> f32 -> bf16; combine in
    f32 in slot order), then masked by the route."""
    X = _f(x).double()
    T = X.shape[0]
    E = wg.shape[0]
    ys = []
    for e in range(E):
        g = (X @ _f(wg[e]).double()).float().double()
        u = (X @ _f(wu[e]).double()).float().double()
        s = g * torch.from_numpy(expit(g.numpy()))          # silu via scipy's logistic
        h = _bf16_bits_t((s * u).float())
        y = _bf16_bits_t((_f(h).double() @ _f(wd[e]).double()).float())
        ys.append(y)
    ys = np.stack(ys)                                      # [E, T, H]
    k = ids.shape[1]
    acc = torch.zeros((T, ys.shape[2]), dtype=torch.float32)
    for j in range(k):
        yj = _f(ys[ids[:, j], np.arange(T)])
        acc = acc + torch.from_numpy(w[:, j]).float()[:, None] * yj
    return _bf16_bits_t(acc), ys


def test_up_row_one_hot_closed_form(oracle_mod):
    rng = np.random.default_rng(11)
    H, I = 64, 48
    wg = moe_inputs._to_bf16_bits(rng.standard_normal((H, I)).astype(np.float32) * 3)
    wu = moe_inputs._to_bf16_bits(rng.standard_normal((H, I)).astype(np.float32))
    for h0 in (0, 17, H - 1):
        x = np.zeros(H, np.uint16)
        x[h0] = 0x3F80                                  # 1.0
        h = oracle_mod.expert_up_row(x, wg, wu)
        g = _f(wg[h0]).double().numpy()
        u = _f(wu[h0]).double().numpy()
        want = _bf16_bits_t(torch.from_numpy(g * expit(g) * u).float())
        assert np.array_equal(h, want)


def test_up_row_silu_special_values(oracle_mod):
    H, I = 8, 4
    x = np.zeros(H, np.uint16)
    x[0] = 0x3F80
    wg = np.zeros((H, I), np.uint16)
    wu = np.zeros((H, I), np.uint16)
    # g = [0, 10, -10, 1], u = 1
    wg[0] = [0x0000, 0x4120, 0xC120, 0x3F80]
    wu[0] = [0x3F80] * 4
    h = oracle_mod.expert_up_row(x, wg, wu)
    vals = _f(h).numpy()
    assert vals[0] == 0.0
    assert vals[1] == 10.0                               # 10/(1+e^-10) = 9.99955 -> bf16 10.0
    np.testing.assert_allclose(vals[2], -10 * expit(-10), rtol=4e-3)
    np.testing.assert_allclose(vals[3], expit(1.0), rtol=4e-3)


def test_down_row_one_hot_is_weight_row(oracle_mod):
    rng = np.random.default_rng(12)
    I, H = 40, 72
    wd = moe_inputs._to_bf16_bits(rng.standard_normal((I, H)).astype(np.float32))
    for i0 in (0, 5, I - 1):
        h = np.zeros(I, np.uint16)
        h[i0] = 0x3F80
        assert np.array_equal(oracle_mod.expert_down_row(h, wd), wd[i0])
        h[i0] = 0x4000                                   # 2.0 doubles the row exactly
        assert np.array_equal(_f(oracle_mod.expert_down_row(h, wd)).numpy(), 2 * _f(wd[i0]).numpy())


def test_dense_swiglu_k1_E1(oracle_mod):
    T, H, I = 96, 128, 256
    logits, x, wg, wu, wd = _small_layer(T, H, I, 1, 1, 5)
    res = oracle_mod.layer(logits, x, wg, wu, wd, 1)
    assert np.all(res.route.topk_w == 1.0)
    X = _f(x).float()
    ref = torch.nn.functional.silu(X @ _f(wg[0])) * (X @ _f(wu[0]))
    ref = _f(_bf16_bits_t(ref)) @ _f(wd[0])
    got = _f(res.out)
    err = (got - ref).abs()
    assert torch.all(err <= 1e-2 + 1e-2 * ref.abs())
    assert (err.norm() / ref.norm()).item() < 5e-3


def test_grouped_path_matches_dense_brute_force(oracle_mod):
    T, H, I, E, k = 64, 128, 128, 6, 3
    logits, x, wg, wu, wd = _small_layer(T, H, I, E, k, 9)
    res = oracle_mod.layer(logits, x, wg, wu, wd, k)
    ref_out, ys = _dense_reference(logits, x, wg, wu, wd, res.route.topk_ids, res.route.topk_w)
    # float64 sums in another order may flip a float32/bf16 rounding at most
    # rarely, and then by one unit
    d = _ulp_diff(res.out, ref_out)
    assert d.max() <= 1 and (d > 0).mean() < 1e-3
    # the permuted rows hold exactly the dense expert outputs of their token
    r = res.route
    real = np.nonzero(r.gather_idx >= 0)[0]
    e_of = r.block_expert[real // 128]
    dy = _ulp_diff(res.Y[real], ys[e_of, r.gather_idx[real]])
    assert dy.max() <= 1 and (dy > 0).mean() < 1e-3


def test_token_path_equals_grouped_path(oracle_mod):
    T, H, I, E, k = 128, 256, 512, 8, 2
    logits, x, wg, wu, wd = _small_layer(T, H, I, E, k, 1001)
    res = oracle_mod.layer(logits, x, wg, wu, wd, k)
    toks = np.array([0, 1, 63, 64, 127], dtype=np.int32)
    out, hs, ys = oracle_mod.tokens_out(toks, res.route.topk_ids, res.route.topk_w,
                                        x, wg, wu, wd, want_rows=True)
    assert np.array_equal(out, res.out[toks])
    rows = res.route.scatter_idx[toks]
    assert np.array_equal(ys, res.Y[rows])
    assert np.array_equal(hs, res.h[rows])


def test_identical_experts_combine_to_one_expert(oracle_mod):
    T, H, I, E, k = 50, 128, 128, 4, 3
    logits, x, wg, wu, wd = _small_layer(T, H, I, E, k, 21)
    wg[:] = wg[0]
    wu[:] = wu[0]
    wd[:] = wd[0]
    res = oracle_mod.layer(logits, x, wg, wu, wd, k)
    single = oracle_mod.layer(np.zeros((T, 1), np.float32), x, wg[:1], wu[:1], wd[:1], 1)
    # sum_j w_j = 1 up to float32 rounding, so out equals y up to one bf16 unit
    d = _ulp_diff(res.out, single.out)
    assert d.max() <= 1
    assert (d == 0).mean() > 0.95


def test_k_equals_E_full_mixture(oracle_mod):
    from scipy.special import softmax
    T, H, I, E = 40, 128, 128, 4
    logits, x, wg, wu, wd = _small_layer(T, H, I, E, E, 31)
    res = oracle_mod.layer(logits, x, wg, wu, wd, E)
    p = softmax(logits.astype(np.float64), axis=1)
    ys = np.stack([oracle_mod.layer(np.zeros((T, 1), np.float32), x, wg[e:e + 1], wu[e:e + 1],
                                    wd[e:e + 1], 1).out for e in range(E)])   # [E, T, H]
    mix = np.einsum("te,eth->th", p, _f(ys).double().numpy())
    got = _f(res.out).double().numpy()
    assert np.all(np.abs(got - mix) <= 1e-2 + 1e-2 * np.abs(mix))


def test_scaling_w_down_by_two_doubles_output(oracle_mod):
    T, H, I, E, k = 32, 128, 128, 4, 2
    logits, x, wg, wu, wd = _small_layer(T, H, I, E, k, 41)
    a = oracle_mod.layer(logits, x, wg, wu, wd, k)
    wd2 = _bf16_bits_t(_f(wd) * 2)
    b = oracle_mod.layer(logits, x, wg, wu, wd2, k)
    assert np.array_equal(_f(b.out).numpy(), 2 * _f(a.out).numpy())
    assert np.array_equal(a.h, b.h)


def test_padding_rows_untouched_and_combine_ignores_them(oracle_mod):
    T, H, I, E, k = 10, 128, 128, 3, 1
    logits, x, wg, wu, wd = _small_layer(T, H, I, E, k, 51)
    res = oracle_mod.layer(logits, x, wg, wu, wd, k)
    pad = res.route.gather_idx < 0
    assert pad.sum() == res.route.num_blocks * 128 - T * k
    assert np.all(res.h[pad] == 0) and np.all(res.Y[pad] == 0)
    # with k=1 each output row is its single expert row (weight exactly 1)
    assert np.array_equal(res.out, res.Y[res.route.scatter_idx[:, 0]])
