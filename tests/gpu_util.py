"""Helpers shared by the GPU parity tests: host<->device transfers of bf16 bit
arrays, the parity tolerances and workload-shaped input builders."""
from __future__ import annotations

import numpy as np
import pytest

# Layer tolerance: |gpu - oracle| <= ATOL + RTOL*|oracle| elementwise and a
# relative Frobenius error <= FRO.
ATOL = 1e-2
RTOL = 1e-2
FRO = 5e-3
# topk_w: the GPU forms exp in float32 (l - max rounded to float32, expf,
# float32 sums over the k picks); the oracle rounds an exact value once.
# Worst case is a few ulps; this bound is 8 ulps of the value.
W_ULPS = 8


_built = False


def need_gpu():
    """Skips without a CUDA device; otherwise makes sure the CUDA library is
    built (in-tree) and returns torch."""
    global _built
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if not _built:
        from combine_moe_route_04_gb300 import _build
        _build.build()
        _built = True
    return torch


def to_dev_bf16(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(torch.bfloat16).cuda()


def to_dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host_u16(t) -> np.ndarray:
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def f32(bits) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def assert_close_layer(got_bits, ref_bits, what="out"):
    g = f32(got_bits).astype(np.float64)
    r = f32(ref_bits).astype(np.float64)
    assert np.all(np.isfinite(g)), "%s: non-finite GPU values" % what
    err = np.abs(g - r)
    bad = err > ATOL + RTOL * np.abs(r)
    if bad.any():
        idx = np.argwhere(bad)[:8]
        raise AssertionError("%s: %d elements outside |d| <= %g + %g|ref|; first %s, max err %g"
                             % (what, int(bad.sum()), ATOL, RTOL, idx.tolist(), err.max()))
    fro = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)
    assert fro <= FRO, "%s: relative Frobenius error %g > %g" % (what, fro, FRO)
    return err.max(), fro


def assert_rows_close(got_bits, ref_bits, what):
    """Row-wise report (a swapped or shifted row fails with its index)."""
    g = f32(got_bits).astype(np.float64)
    r = f32(ref_bits).astype(np.float64)
    err = np.abs(g - r) - (ATOL + RTOL * np.abs(r))
    bad_rows = np.nonzero((err > 0).any(axis=-1))[0]
    assert bad_rows.size == 0, "%s: rows %s out of tolerance (of %d)" % (what, bad_rows[:16].tolist(), g.shape[0])
    return assert_close_layer(got_bits, ref_bits, what)


def ulp_dist_f32(a, b) -> np.ndarray:
    a = np.asarray(a, np.float32).view(np.int32).astype(np.int64)
    b = np.asarray(b, np.float32).view(np.int32).astype(np.int64)
    a = np.where(a < 0, -(a & 0x7FFFFFFF), a)
    b = np.where(b < 0, -(b & 0x7FFFFFFF), b)
    return np.abs(a - b)


def assert_close_whole(got_bits, ref_bits, what, chunk_rows=4096):
    """The layer tolerance over a whole 2-D array, in row chunks (bounded host
    memory): every element within ATOL + RTOL*|ref|, the first bad rows
    reported by index, and the relative Frobenius error over the WHOLE array
    (accumulated across chunks) <= FRO.  Returns (max |err|, rel. Frobenius)."""
    got_bits = np.asarray(got_bits)
    ref_bits = np.asarray(ref_bits)
    assert got_bits.shape == ref_bits.shape, "%s: shape %s vs %s" % (what, got_bits.shape, ref_bits.shape)
    n = got_bits.shape[0]
    d2 = 0.0
    r2 = 0.0
    max_err = 0.0
    bad_rows = []
    for r0 in range(0, n, chunk_rows):
        g = f32(got_bits[r0:r0 + chunk_rows]).astype(np.float64)
        r = f32(ref_bits[r0:r0 + chunk_rows]).astype(np.float64)
        assert np.all(np.isfinite(g)), "%s: non-finite GPU values in rows %d.." % (what, r0)
        err = np.abs(g - r)
        bad = (err > ATOL + RTOL * np.abs(r)).any(axis=-1)
        if bad.any() and len(bad_rows) < 16:
            bad_rows.extend((r0 + np.nonzero(bad)[0][:16]).tolist())
        max_err = max(max_err, float(err.max()) if err.size else 0.0)
        d2 += float(np.sum((g - r) ** 2))
        r2 += float(np.sum(r * r))
    assert not bad_rows, "%s: rows %s out of tolerance (of %d), max err %g" % (what, bad_rows[:16], n, max_err)
    fro = (d2 ** 0.5) / max(r2 ** 0.5, 1e-30)
    assert fro <= FRO, "%s: relative Frobenius error %g > %g" % (what, fro, FRO)
    return max_err, fro
