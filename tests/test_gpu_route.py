"""GPU parity of moe_route against the oracle: picks, counts, padded offsets,
block table and permutation bit-exact; weights within a few float32 ulps."""
import numpy as np
import pytest

import moe_inputs
from gpu_util import W_ULPS, need_gpu, to_dev, ulp_dist_f32

pytestmark = pytest.mark.gpu


def run_route(logits, k):
    torch = need_gpu()
    import combine_moe_route_04_gb300 as moe
    T, E = logits.shape
    s = moe.shape(T, 128, 128, E, k)
    bufs = moe.alloc_route_outputs(s)
    bufs["gather_idx"].fill_(-7)          # sentinel: rows the route must not touch
    ws = moe.alloc_workspace(s)
    moe.moe_route(s, to_dev(logits), bufs["topk_ids"], bufs["topk_w"], bufs["counts"],
                  bufs["off_pad"], bufs["block_expert"], bufs["num_blocks"], bufs["gather_idx"],
                  bufs["scatter_idx"], ws)
    assert moe.last_device_status(ws) == 0
    return {k_: v.cpu().numpy() for k_, v in bufs.items()}


def check_route(logits, k, oracle_mod):
    got = run_route(logits, k)
    ref = oracle_mod.route(logits, k)
    nb = int(got["num_blocks"][0])
    assert nb == ref.num_blocks
    assert np.array_equal(got["topk_ids"], ref.topk_ids)
    assert np.array_equal(got["counts"], ref.counts)
    assert np.array_equal(got["off_pad"], ref.off_pad)
    assert np.array_equal(got["block_expert"][:nb], ref.block_expert)
    assert np.array_equal(got["gather_idx"][:nb * 128], ref.gather_idx)
    assert np.all(got["gather_idx"][nb * 128:] == -7)
    assert np.array_equal(got["scatter_idx"], ref.scatter_idx)
    d = ulp_dist_f32(got["topk_w"], ref.topk_w)
    assert d.max() <= W_ULPS, "topk_w off by %d ulps" % d.max()
    return got, ref


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_route_workloads(oracle_mod, n):
    cfg = moe_inputs.config(n)
    logits = moe_inputs.make_logits(cfg.T, cfg.E, cfg.seed, cfg.logit_bias)
    got, ref = check_route(logits, cfg.k, oracle_mod)
    if n == 4:
        assert (ref.counts == 0).sum() > 0     # skewed: several experts empty


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (1, 8, 8), (33, 256, 16), (4097, 64, 8), (31, 5, 5),
                                   (2, 256, 1),
                                   (1 << 18, 256, 16),   # E and k at their limits: 4.2 M rows, 8192 chunks
                                   (1 << 22, 8, 2)])     # T at its limit: 131 072 chunks per expert scan
def test_route_edge_shapes(oracle_mod, T, E, k):
    rng = np.random.default_rng(T + 17 * E + k)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    check_route(logits, k, oracle_mod)


def test_route_ties_integer_logits(oracle_mod):
    rng = np.random.default_rng(5)
    logits = rng.integers(-1, 2, size=(1000, 16)).astype(np.float32)
    check_route(logits, 4, oracle_mod)


def test_route_exact_block_boundaries(oracle_mod):
    # e0 gets exactly 128 rows, e1 129 rows, e2 none, e3 one row
    T, E = 258, 4
    logits = np.full((T, E), -10.0, dtype=np.float32)
    logits[:128, 0] = 10
    logits[128:257, 1] = 10
    logits[257, 3] = 10
    got, ref = check_route(logits, 1, oracle_mod)
    assert ref.counts.tolist() == [128, 129, 0, 1]
    assert ref.off_pad.tolist() == [0, 128, 384, 384, 512]
