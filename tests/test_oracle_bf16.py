"""Pins of the oracle's bfloat16 rounding (round to nearest, ties to even)
against torch's CPU float32 -> bfloat16 conversion (a library routine) and
against hand-worked bit patterns."""
import numpy as np
import pytest
import torch


def _torch_bf16_bits(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _f32(bits):
    return np.array(bits, dtype=np.uint32).view(np.float32)


def test_bf16_hand_worked(oracle_mod):
    cases = {
        0x3F800000: 0x3F80,  # 1.0 exact
        0x3F808000: 0x3F80,  # halfway, kept part even -> stays
        0x3F818000: 0x3F82,  # halfway, kept part odd -> rounds up to even
        0x3F808001: 0x3F81,  # just above half -> up
        0x3F807FFF: 0x3F80,  # just below half -> down
        0x3FFF8000: 0x4000,  # carry into the exponent: 1.99609375+ -> 2.0
        0x7F7FFFFF: 0x7F80,  # max finite rounds to +inf
        0x80000000: 0x8000,  # -0
        0x00000001: 0x0000,  # smallest subnormal rounds to 0
        0x00018000: 0x0002,  # subnormal tie, kept odd -> up
        0x7F800000: 0x7F80,  # +inf
        0xFF800000: 0xFF80,  # -inf
    }
    got = oracle_mod.bf16_from_f32(_f32(list(cases.keys())))
    assert [int(g) for g in got] == list(cases.values())
    nan = oracle_mod.bf16_from_f32(_f32([0x7FC00001, 0xFF800001]))
    assert all((int(n) & 0x7F80) == 0x7F80 and (int(n) & 0x7F) != 0 for n in nan)


def test_bf16_matches_torch_on_random_bits(oracle_mod):
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2**32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    # exclude NaNs (payload conventions differ), keep inf/subnormal/normal
    f = bits.view(np.float32)
    f = f[~np.isnan(f)]
    assert np.array_equal(oracle_mod.bf16_from_f32(f), _torch_bf16_bits(f))


def test_bf16_matches_torch_on_ties(oracle_mod):
    rng = np.random.default_rng(8)
    hi = rng.integers(0, 0x7F7F, size=100_000, dtype=np.uint32)
    bits = (hi << 16) | 0x8000          # exact halfway points
    f = bits.view(np.float32)
    assert np.array_equal(oracle_mod.bf16_from_f32(f), _torch_bf16_bits(f))


def test_f32_from_bf16_roundtrip(oracle_mod):
    b = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    f = oracle_mod.f32_from_bf16(b)
    ok = ~np.isnan(f)
    assert np.array_equal(oracle_mod.bf16_from_f32(f[ok]), b[ok])
