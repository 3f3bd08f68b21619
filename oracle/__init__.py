"""CPU oracle of the MoE expert layer -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package.  It shares no code with the CUDA
library: the arithmetic lives in ``moe_oracle.c`` (plain C, double
accumulation, compiled with gcc and ``-ffp-contract=off``) and this module
only marshals numpy arrays into it.

Every function is pinned by the ``-m "not gpu"`` tests (brute force on tiny
inputs, closed forms, library special cases, invariants); no page prints a
numeric example of the layer, so none is pinned to a printed value.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")

ROW_BLOCK = 128


def build_oracle(force: bool = False) -> str:
    """Compile moe_oracle.c into libmoe_oracle.so (gcc, OpenMP)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        build_oracle()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i32, i64 = ctypes.c_int32, ctypes.c_int64
        lib.oracle_bf16_from_f32.restype = ctypes.c_uint16
        lib.oracle_bf16_from_f32.argtypes = [ctypes.c_float]
        lib.oracle_f32_from_bf16.restype = ctypes.c_float
        lib.oracle_f32_from_bf16.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_from_f32_array.argtypes = [i64, P, P]
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        lib.oracle_route_select.argtypes = [ctypes.c_int] * 3 + [P, P, P]
        lib.oracle_max_blocks.restype = i64
        lib.oracle_max_blocks.argtypes = [ctypes.c_int] * 3
        lib.oracle_route_permute.restype = ctypes.c_int
        lib.oracle_route_permute.argtypes = [ctypes.c_int] * 3 + [P] * 7 + [i64]
        lib.oracle_expert_up_row.argtypes = [ctypes.c_int] * 2 + [P] * 5
        lib.oracle_expert_down_row.argtypes = [ctypes.c_int] * 2 + [P] * 4
        lib.oracle_grouped_up.argtypes = [ctypes.c_int] * 4 + [i32] + [P] * 6
        lib.oracle_grouped_down.argtypes = [ctypes.c_int] * 3 + [i32] + [P] * 5
        lib.oracle_combine.argtypes = [ctypes.c_int] * 3 + [P] * 4
        lib.oracle_tokens_out.argtypes = ([ctypes.c_int, P] + [ctypes.c_int] * 3
                                          + [P] * 9)
        _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a):
    return np.ascontiguousarray(a, dtype=np.uint16)


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


# ------------------------------------------------------------------ bf16

def bf16_from_f32(a) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.uint16)
    _load().oracle_bf16_from_f32_array(a.size, _p(a), _p(out))
    return out


def f32_from_bf16(b) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------------ route

def max_blocks(T: int, E: int, k: int) -> int:
    return int(_load().oracle_max_blocks(T, E, k))


def route_select(logits: np.ndarray, k: int):
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    _load().oracle_route_select(T, E, k, _p(logits), _p(ids), _p(w))
    return ids, w


@dataclass
class Route:
    topk_ids: np.ndarray     # [T, k] int32
    topk_w: np.ndarray       # [T, k] float32
    counts: np.ndarray       # [E] int32
    off_pad: np.ndarray      # [E+1] int32
    block_expert: np.ndarray  # [num_blocks] int32
    num_blocks: int
    gather_idx: np.ndarray   # [num_blocks*128] int32
    scatter_idx: np.ndarray  # [T, k] int32


def route_permute(topk_ids: np.ndarray, E: int) -> tuple:
    ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    T, k = ids.shape
    mb = max_blocks(T, E, k)
    counts = np.empty(E, dtype=np.int32)
    off_pad = np.empty(E + 1, dtype=np.int32)
    block_expert = np.empty(max(mb, 1), dtype=np.int32)
    nb = np.zeros(1, dtype=np.int32)
    gather = np.empty(max(mb, 1) * ROW_BLOCK, dtype=np.int32)
    scatter = np.empty((T, k), dtype=np.int32)
    rc = _load().oracle_route_permute(T, E, k, _p(ids), _p(counts), _p(off_pad),
                                      _p(block_expert), _p(nb), _p(gather),
                                      _p(scatter), mb * ROW_BLOCK)
    if rc != 0:
        raise RuntimeError("oracle_route_permute: capacity exceeded")
    n = int(nb[0])
    return counts, off_pad, block_expert[:n].copy(), n, gather[:n * ROW_BLOCK].copy(), scatter


def route(logits: np.ndarray, k: int) -> Route:
    T, E = logits.shape
    ids, w = route_select(logits, k)
    counts, off_pad, be, n, gather, scatter = route_permute(ids, E)
    return Route(ids, w, counts, off_pad, be, n, gather, scatter)


# ------------------------------------------------------------- expert FFN

def expert_up_row(x, wg_e, wu_e):
    x, wg_e, wu_e = _u16(x), _u16(wg_e), _u16(wu_e)
    H, I = wg_e.shape
    h = np.empty(I, dtype=np.uint16)
    acc = np.empty(2 * I, dtype=np.float64)
    _load().oracle_expert_up_row(H, I, _p(x), _p(wg_e), _p(wu_e), _p(h), _p(acc))
    return h


def expert_down_row(h, wd_e):
    h, wd_e = _u16(h), _u16(wd_e)
    I, H = wd_e.shape
    y = np.empty(H, dtype=np.uint16)
    acc = np.empty(H, dtype=np.float64)
    _load().oracle_expert_down_row(H, I, _p(h), _p(wd_e), _p(y), _p(acc))
    return y


def grouped_up(X, r: Route, Wg, Wu):
    X, Wg, Wu = _u16(X), _u16(Wg), _u16(Wu)
    T, H = X.shape
    E, _, I = Wg.shape
    h = np.zeros((r.num_blocks * ROW_BLOCK, I), dtype=np.uint16)
    be = np.ascontiguousarray(r.block_expert, dtype=np.int32)
    g = np.ascontiguousarray(r.gather_idx, dtype=np.int32)
    _load().oracle_grouped_up(T, H, I, E, r.num_blocks, _p(be), _p(g),
                              _p(X), _p(Wg), _p(Wu), _p(h))
    return h


def grouped_down(h, r: Route, Wd):
    h, Wd = _u16(h), _u16(Wd)
    E, I, H = Wd.shape
    Y = np.zeros((r.num_blocks * ROW_BLOCK, H), dtype=np.uint16)
    be = np.ascontiguousarray(r.block_expert, dtype=np.int32)
    g = np.ascontiguousarray(r.gather_idx, dtype=np.int32)
    _load().oracle_grouped_down(H, I, E, r.num_blocks, _p(be), _p(g), _p(h),
                                _p(Wd), _p(Y))
    return Y


def combine(Y, scatter_idx, topk_w):
    Y = _u16(Y)
    s = np.ascontiguousarray(scatter_idx, dtype=np.int32)
    w = np.ascontiguousarray(topk_w, dtype=np.float32)
    T, k = s.shape
    H = Y.shape[1]
    out = np.empty((T, H), dtype=np.uint16)
    _load().oracle_combine(T, H, k, _p(Y), _p(s), _p(w), _p(out))
    return out


@dataclass
class LayerResult:
    route: Route
    h: np.ndarray     # [num_blocks*128, I] bf16 bits (padding rows zero)
    Y: np.ndarray     # [num_blocks*128, H] bf16 bits (padding rows zero)
    out: np.ndarray   # [T, H] bf16 bits


def layer(logits, X, Wg, Wu, Wd, k: int) -> LayerResult:
    """The whole layer, step by step: route, grouped up, grouped down, combine."""
    r = route(logits, k)
    h = grouped_up(X, r, Wg, Wu)
    Y = grouped_down(h, r, Wd)
    out = combine(Y, r.scatter_idx, r.topk_w)
    return LayerResult(r, h, Y, out)


def tokens_out(tokens, topk_ids, topk_w, X, Wg, Wu, Wd, want_rows: bool = False):
    """Layer output of selected tokens, token by token (no permutation).

    topk_ids/topk_w are the full [T, k] route; returns out [n, H] and, with
    want_rows, the per-slot rows h [n, k, I] and y [n, k, H]."""
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    ids = np.ascontiguousarray(np.asarray(topk_ids)[tokens], dtype=np.int32)
    w = np.ascontiguousarray(np.asarray(topk_w)[tokens], dtype=np.float32)
    X, Wg, Wu, Wd = _u16(X), _u16(Wg), _u16(Wu), _u16(Wd)
    n = tokens.shape[0]
    k = ids.shape[1]
    E, H, I = Wg.shape
    out = np.empty((n, H), dtype=np.uint16)
    hs = np.empty((n, k, I), dtype=np.uint16) if want_rows else None
    ys = np.empty((n, k, H), dtype=np.uint16) if want_rows else None
    _load().oracle_tokens_out(n, _p(tokens), H, I, k, _p(ids), _p(w), _p(X),
                              _p(Wg), _p(Wu), _p(Wd), _p(out),
                              _p(hs) if want_rows else None,
                              _p(ys) if want_rows else None)
    if want_rows:
        return out, hs, ys
    return out
