"""Pins of the oracle's routing: hand-worked golden case, brute force over all
k-subsets on tiny inputs, the k = E special case against scipy's softmax, tie
handling with integer logits, and the permutation invariants."""
import itertools
import math
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            rows.setdefault(key, []).append(vals)
    return rows


def test_route_hand_worked_golden(oracle_mod):
    g = _read_golden("route_tiny.txt")
    logits = np.array([[float(v) for v in r] for r in g["logits"]], dtype=np.float32)
    T, E = logits.shape
    k = 2
    r = oracle_mod.route(logits, k)
    assert r.topk_ids.tolist() == [[int(v) for v in row] for row in g["topk_ids"]]
    want_w = np.array([[float(v) for v in row] for row in g["topk_w"]], dtype=np.float32)
    assert np.array_equal(r.topk_w, want_w)
    assert r.counts.tolist() == [int(v) for v in g["counts"][0]]
    assert r.off_pad.tolist() == [int(v) for v in g["off_pad"][0]]
    assert r.num_blocks == int(g["num_blocks"][0][0])
    assert r.block_expert.tolist() == [int(v) for v in g["block_expert"][0]]
    assert r.scatter_idx.tolist() == [[int(v) for v in row] for row in g["scatter_idx"]]
    want_gather = np.full(r.num_blocks * 128, -1, dtype=np.int32)
    for item in g["gather"][0]:
        row, tok = item.split(":")
        want_gather[int(row)] = int(tok)
    assert np.array_equal(r.gather_idx, want_gather)


def _brute_topk(l, k):
    """Best k-subset by brute force: the subset whose keys (logit, -index),
    sorted descending, are lexicographically largest; slots in that order."""
    E = len(l)
    best = None
    for sub in itertools.combinations(range(E), k):
        keys = sorted(((float(l[e]), -e) for e in sub), reverse=True)
        if best is None or keys > best:
            best = keys
    return [-key[1] for key in best]


def _weights_cancelled_form(l, ids):
    # w_j = exp(l_j) / sum_{j' in picks} exp(l_j'): the softmax denominator
    # cancels in the renormalisation; computed with exact summation.
    m = max(float(l[e]) for e in ids)
    ex = [math.exp(float(l[e]) - m) for e in ids]
    s = math.fsum(ex)
    return [x / s for x in ex]


@pytest.mark.parametrize("E,k", [(1, 1), (2, 1), (3, 2), (5, 3), (6, 6), (7, 2), (8, 4)])
def test_route_select_brute_force(oracle_mod, E, k):
    rng = np.random.default_rng(100 + 10 * E + k)
    T = 64
    # small-integer logits force many ties; half the tokens use continuous values
    logits = np.where(rng.random((T, E)) < 0.5,
                      rng.integers(-2, 3, size=(T, E)).astype(np.float32),
                      rng.standard_normal((T, E)).astype(np.float32))
    ids, w = oracle_mod.route_select(logits, k)
    for t in range(T):
        want = _brute_topk(logits[t], k)
        assert ids[t].tolist() == want, (t, logits[t])
        ww = _weights_cancelled_form(logits[t], want)
        np.testing.assert_allclose(w[t], np.array(ww, dtype=np.float32), rtol=2e-7, atol=0)


def test_route_weights_k_equals_E_is_softmax(oracle_mod):
    from scipy.special import softmax
    rng = np.random.default_rng(3)
    T, E = 200, 16
    logits = (3 * rng.standard_normal((T, E))).astype(np.float32)
    ids, w = oracle_mod.route_select(logits, E)
    p = softmax(logits.astype(np.float64), axis=1)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-logits[t, e], e))
        assert ids[t].tolist() == order
        np.testing.assert_allclose(w[t], p[t, order].astype(np.float32), rtol=3e-7, atol=1e-30)
        assert abs(float(np.sum(w[t].astype(np.float64))) - 1.0) < 1e-6


def test_route_ties_integer_logits(oracle_mod):
    logits = np.array([[1, 3, 3, 2, 3]], dtype=np.float32)
    assert oracle_mod.route_select(logits, 2)[0].tolist() == [[1, 2]]
    assert oracle_mod.route_select(logits, 4)[0].tolist() == [[1, 2, 4, 3]]
    assert oracle_mod.route_select(logits, 5)[0].tolist() == [[1, 2, 4, 3, 0]]
    w = oracle_mod.route_select(logits, 3)[1]
    assert np.array_equal(w, np.full((1, 3), np.float32(1 / 3)))


def test_route_large_logits_no_overflow(oracle_mod):
    logits = np.array([[1000.0, 999.0, -1000.0, 0.0]], dtype=np.float32)
    ids, w = oracle_mod.route_select(logits, 2)
    assert ids.tolist() == [[0, 1]]
    e = math.exp(-1.0)
    np.testing.assert_allclose(w[0], [1 / (1 + e), e / (1 + e)], rtol=2e-7)


def check_permutation_invariants(T, E, k, ids, counts, off_pad, block_expert, nb, gather, scatter):
    R = T * k
    assert counts.sum() == R
    assert np.array_equal(counts, np.bincount(ids.ravel(), minlength=E))
    assert off_pad[0] == 0 and np.all(off_pad % 128 == 0)
    padded = np.diff(off_pad)
    assert np.array_equal(padded, (counts + 127) // 128 * 128)
    assert nb == off_pad[E] // 128
    assert np.all(np.diff(block_expert) >= 0)
    assert np.array_equal(np.bincount(block_expert, minlength=E), padded // 128)
    # bijection between real rows and (t, j)
    flat = scatter.ravel()
    assert len(np.unique(flat)) == R
    assert np.all(gather[flat] == np.repeat(np.arange(T), k))
    assert (gather >= 0).sum() == R
    # each row lies inside its expert's padded range, real rows first
    e_of = ids.ravel()
    assert np.all(flat >= off_pad[e_of]) and np.all(flat < off_pad[e_of] + counts[e_of])
    # stable: within an expert, rows ascend with the token
    for e in range(E):
        rows = np.arange(off_pad[e], off_pad[e] + counts[e])
        assert np.all(np.diff(gather[rows]) > 0)


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (1, 8, 8), (37, 5, 2), (128, 8, 2), (300, 2, 1),
                                   (1000, 64, 8), (513, 256, 16)])
def test_route_permutation_invariants(oracle_mod, T, E, k):
    rng = np.random.default_rng(T * 7 + E * 3 + k)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    if T == 300:
        logits[:, 0] += 100.0   # every token to expert 0: three blocks, ragged tail
    r = oracle_mod.route(logits, k)
    check_permutation_invariants(T, E, k, r.topk_ids, r.counts, r.off_pad, r.block_expert,
                                 r.num_blocks, r.gather_idx, r.scatter_idx)
    assert r.num_blocks <= oracle_mod.max_blocks(T, E, k)
    if T == 300:
        assert r.counts.tolist() == [300, 0] and r.off_pad.tolist() == [0, 384, 384]
        assert r.block_expert.tolist() == [0, 0, 0]


def test_max_blocks_is_tight(oracle_mod):
    # every expert gets exactly one routed row: E blocks of 1 row each
    T, E, k = 8, 8, 1
    logits = np.full((T, E), -5.0, dtype=np.float32)
    for t in range(T):
        logits[t, t] = 5.0
    r = oracle_mod.route(logits, k)
    assert r.num_blocks == E == oracle_mod.max_blocks(T, E, k)
