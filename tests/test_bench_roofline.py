"""The benchmark's roofline arithmetic (CPU only).

The layer's algorithmic bytes and FLOPs are those of the per-step model:
route T*E*4 + 12*T*k + 4*R_pad; gate/up touched*2*H*I*2 + T*H*2 + R*I*2;
down touched*I*H*2 + R*I*2 + R*H*2; combine R*H*2 + 8*T*k + T*H*2; FLOPs
6*R*H*I with R = T*k.  Pinned here to hand-worked values of the
pages-shaped workload (2.82 GB, 618.5 GFLOP, 416 us at the 6.78 TB/s copy
rate), and the bound and fraction to the slower of the two floors."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
import moe_inputs  # noqa: E402

PEAKS = {"hbm_gbs": 6782.8, "bf16_tflops": 1897.5, "bf16_tflops_sustained": 1708.7}


def test_layer_bytes_pages_shaped():
    cfg = moe_inputs.config(2)       # T=2048, H=4096, I=1536, E=64, k=8
    # the workload's routing fills 158 blocks of 128 rows (R_pad = 20224)
    b = bench.layer_bytes(cfg, touched=64, r_pad=20224)
    # worked by hand from the formulas in the docstring
    assert b["route"] == 2048 * 64 * 4 + 12 * 2048 * 8 + 4 * 20224 == 801792
    assert b["up"] == 64 * 2 * 4096 * 1536 * 2 + 2048 * 4096 * 2 + 16384 * 1536 * 2 == 1677721600
    assert b["down"] == 64 * 1536 * 4096 * 2 + 16384 * 1536 * 2 + 16384 * 4096 * 2 == 989855744
    assert b["combine"] == 16384 * 4096 * 2 + 8 * 2048 * 8 + 2048 * 4096 * 2 == 151126016
    assert abs(sum(b.values()) / 1e9 - 2.8195) < 1e-4
    assert bench.layer_flops(cfg) == 6 * 16384 * 4096 * 1536 == 618475290624


def test_layer_roofline_bound_and_fraction():
    cfg = moe_inputs.config(2)
    r = bench.layer_roofline(cfg, 64, 20224, ms_step=0.5406, pk=PEAKS, pk_src="measured")
    # bytes at 6782.8 GB/s: 415.7 us; FLOPs at 1708.7 TFLOP/s: 362.0 us -> HBM-bound
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["hbm_floor_us"] == pytest.approx(2819505152 / 6782.8e9 * 1e6, rel=1e-9)
    assert r["tensor_floor_us"] == pytest.approx(618475290624 / 1708.7e12 * 1e6, rel=1e-9)
    assert r["floor_us"] == pytest.approx(415.68, abs=0.01)
    assert r["frac"] == pytest.approx(415.68 / 540.6, abs=1e-4)
    assert r["achieved"] == pytest.approx(2819505152 / 540.6e-6 / 1e9, rel=1e-9)


def test_layer_roofline_tensor_bound_when_flops_dominate():
    cfg = moe_inputs.config(5)       # T=16384, E=128: the FLOP floor is the larger
    r = bench.layer_roofline(cfg, 128, 139904, ms_step=3.5, pk=PEAKS, pk_src="measured")
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["tensor_floor_us"] > r["hbm_floor_us"]
    assert r["frac"] == pytest.approx(r["tensor_floor_us"] / 3500.0, rel=1e-9)
