"""Seeded synthetic inputs for the MoE expert layer.

This module is shared by the CUDA path's tests/benchmark and by the CPU
oracle, and it holds none of the layer's arithmetic: it only draws the
inputs (router logits, token activations, expert weights) with the shapes
and value distributions of the five workloads below and encodes them as the
bit patterns the layer consumes (float32 logits, bfloat16 activations and
weights stored as raw uint16).

Distributions (one per workload, all synthetic, no dataset):
  * X ~ N(0, 1), rounded to bfloat16 (round-to-nearest-even via torch's CPU
    conversion);
  * W_gate, W_up ~ N(0, 1/H) and W_down ~ N(0, 1/I) ("N(0, 1/fan_in)" with
    fan_in the reduction length of each projection), rounded to bfloat16;
  * router logits ~ N(0, 1) float32; the skewed workload adds a per-expert
    bias b_e = 3 * ln(1 / (e + 1)).

Every tensor (and every expert slice of a weight tensor) is drawn from its own
PCG64 stream keyed by (seed, tensor id, expert), so the values do not depend
on the thread count used to draw them.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import math
import os

import numpy as np

__all__ = ["MoEConfig", "CONFIGS", "config", "make_inputs", "make_logits",
           "make_tokens", "make_weights", "max_blocks", "max_rows"]


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int        # tokens
    H: int        # hidden size
    I: int        # expert intermediate size
    E: int        # experts
    k: int        # experts per token
    logit_bias: str = "none"   # "none" | "zipf3" (b_e = 3 ln(1/(e+1)))
    seed: int = 0

    @property
    def shape(self):
        return (self.T, self.H, self.I, self.E, self.k)


# The five synthetic workloads of the layer, numbered 1..5.  Seeds are
# 1000 + workload number.
CONFIGS = {
    1: MoEConfig("tiny", 128, 256, 512, 8, 2, seed=1001),
    2: MoEConfig("pages_shaped_T2048", 2048, 4096, 1536, 64, 8, seed=1002),
    3: MoEConfig("decode_T64", 64, 4096, 1536, 64, 8, seed=1003),
    4: MoEConfig("skewed_T8192", 8192, 4096, 1536, 64, 8, logit_bias="zipf3", seed=1004),
    5: MoEConfig("prefill_T16384", 16384, 4096, 1536, 128, 8, seed=1005),
}


def config(n: int) -> MoEConfig:
    return CONFIGS[n]


def max_blocks(T: int, E: int, k: int) -> int:
    """Upper bound on the number of 128-row expert blocks for any routing.

    sum_e ceil(c_e/128) <= (T*k + 127*min(E, T*k)) / 128.
    """
    R = T * k
    return (R + 127 * min(E, R)) // 128


def max_rows(T: int, E: int, k: int) -> int:
    return 128 * max_blocks(T, E, k)


_TENSOR_IDS = {"logits": 1, "x": 2, "w_gate": 3, "w_up": 4, "w_down": 5}


def _rng(seed: int, tensor: str, part: int = 0) -> np.random.Generator:
    return np.random.default_rng([seed, _TENSOR_IDS[tensor], part])


def _to_bf16_bits(a: np.ndarray) -> np.ndarray:
    import torch  # CPU only: bit-exact round-to-nearest-even conversion
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _normal_bf16(seed, tensor, part, shape, std):
    g = _rng(seed, tensor, part)
    v = g.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        v *= np.float32(std)
    return _to_bf16_bits(v)


def make_logits(T: int, E: int, seed: int, bias: str = "none") -> np.ndarray:
    g = _rng(seed, "logits")
    l = g.standard_normal((T, E), dtype=np.float32)
    if bias == "zipf3":
        b = np.array([3.0 * math.log(1.0 / (e + 1)) for e in range(E)], dtype=np.float64)
        l = (l.astype(np.float64) + b[None, :]).astype(np.float32)
    elif bias != "none":
        raise ValueError(bias)
    return np.ascontiguousarray(l)


def make_tokens(T: int, H: int, seed: int, row_signature: bool = False) -> np.ndarray:
    """X [T, H] as bf16 bits.  With row_signature, row t is scaled by
    (1 + t/1024) before rounding so that a swapped row is visible."""
    g = _rng(seed, "x")
    v = g.standard_normal((T, H), dtype=np.float32)
    if row_signature:
        v *= (1.0 + np.arange(T, dtype=np.float32) / 1024.0)[:, None]
    return _to_bf16_bits(v)


def make_weights(E: int, H: int, I: int, seed: int, threads: int | None = None):
    """(W_gate [E,H,I], W_up [E,H,I], W_down [E,I,H]) as bf16 bits."""
    wg = np.empty((E, H, I), dtype=np.uint16)
    wu = np.empty((E, H, I), dtype=np.uint16)
    wd = np.empty((E, I, H), dtype=np.uint16)
    sg = 1.0 / math.sqrt(H)
    sd = 1.0 / math.sqrt(I)

    def job(args):
        name, e = args
        if name == "w_gate":
            wg[e] = _normal_bf16(seed, name, e, (H, I), sg)
        elif name == "w_up":
            wu[e] = _normal_bf16(seed, name, e, (H, I), sg)
        else:
            wd[e] = _normal_bf16(seed, name, e, (I, H), sd)

    jobs = [(n, e) for n in ("w_gate", "w_up", "w_down") for e in range(E)]
    n = threads or min(32, os.cpu_count() or 1)
    if n <= 1 or len(jobs) == 1:
        for j in jobs:
            job(j)
    else:
        with _cf.ThreadPoolExecutor(n) as ex:
            list(ex.map(job, jobs))
    return wg, wu, wd


def make_inputs(cfg: MoEConfig | int, row_signature: bool = False, seed: int | None = None):
    """All inputs of one workload: dict of numpy arrays."""
    if isinstance(cfg, int):
        cfg = CONFIGS[cfg]
    s = cfg.seed if seed is None else seed
    logits = make_logits(cfg.T, cfg.E, s, cfg.logit_bias)
    x = make_tokens(cfg.T, cfg.H, s, row_signature)
    wg, wu, wd = make_weights(cfg.E, cfg.H, cfg.I, s)
    return {"logits": logits, "x": x, "w_gate": wg, "w_up": wu, "w_down": wd}
