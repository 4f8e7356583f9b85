"""The benchmark's arithmetic on the CPU: the algorithmic work per pass of each workload (FLOPs =
2 R V d; bytes = the operands read once plus O(R) outputs), the roofline fields derived from a
given head time and peaks, and the per-pass loop breakdown from a kernel timeline."""
import math

import pytest

import bench
from workloads import CONFIGS


def test_algorithmic_work_of_the_full_vocabulary_pass():
    cfg = CONFIGS["pass_bf16_v262144_d2816"]
    flops, byts = bench.algorithmic(cfg)
    assert flops == 2 * 256 * 262144 * 2816 == pytest.approx(3.780e11, rel=1e-3)
    w = 262144 * 2816 * 2
    assert w == pytest.approx(1.4764e9, rel=1e-4)
    assert byts == w + 256 * 2816 * 2 + 256 * 17


def test_algorithmic_work_of_the_quantised_heads():
    e4 = CONFIGS["loop_e4m3_v262144_d2816"]
    _, b8 = bench.algorithmic(e4)
    # E4M3 codes + fp32 row scales of W and of h, h codes, outputs
    assert b8 == 262144 * 2816 + 262144 * 4 + 256 * 2816 + 256 * 4 + 256 * 17
    f4 = CONFIGS["pass_nvfp4_v262144_d2816"]
    _, b4 = bench.algorithmic(f4)
    # 4-bit codes, one E4M3 scale per 16 elements, fp32 row scales; bf16 h read once
    assert b4 == 262144 * 2816 / 2 + 262144 * 2816 / 16 + 262144 * 4 + 256 * 2816 * 2 + 256 * 17
    assert b4 == pytest.approx(0.4177e9, rel=1e-3)


PEAKS = {"hbm_gbs": 6500.0, "bf16_tflops": 1700.0, "bf16_tflops_sustained": 1350.0}


def test_roofline_compute_bound_bf16():
    cfg = CONFIGS["pass_bf16_v262144_d2816"]
    flops, byts = bench.algorithmic(cfg)
    head_us = 325.0
    r = {"head_ms": [head_us / 1e3] * 4, "flops": flops, "bytes": byts}
    out = bench.roofline(cfg, r, PEAKS, "measured", step_s=337e-6)
    # t_flop = 3.78e11 / 1.35e15 = 280 us > t_mem = 1.478e9 / 6.5e12 = 227 us: tensor-bound
    assert out["bound"] == "tensor" and out["unit"] == "TFLOP/s"
    assert out["achieved"] == pytest.approx(flops / (head_us * 1e-6) / 1e12)
    assert out["peak"] == 1350.0
    assert out["frac"] == pytest.approx(out["achieved"] / 1350.0)
    assert out["t_roof_us"] == pytest.approx(flops / 1.35e15 * 1e6)
    assert out["hbm_frac"] == pytest.approx(byts / (head_us * 1e-6) / 6.5e12)
    assert out["step_roof_frac"] == pytest.approx(flops / 1.35e15 / 337e-6)
    # datasheet roofline: max(bytes / 8 TB/s, flops / 2.25 PF/s) = the HBM term (184.7 us)
    assert out["datasheet_roof_frac"] == pytest.approx(byts / 8e12 / (head_us * 1e-6))
    assert out["kernel"] == "head_tc2_kernel<0>"


def test_roofline_memory_bound_nvfp4_uses_the_hbm_peak():
    cfg = CONFIGS["pass_nvfp4_v262144_d2816"]
    flops, byts = bench.algorithmic(cfg)
    r = {"head_ms": [0.1175], "flops": flops, "bytes": byts}
    out = bench.roofline(cfg, r, PEAKS, "measured", step_s=130e-6)
    # t_flop at 6 x 1.35 PF/s = 47 us < t_mem = 64 us: HBM-bound
    assert out["bound"] == "hbm" and out["unit"] == "GB/s"
    assert out["achieved"] == pytest.approx(byts / 117.5e-6 / 1e9)
    assert out["frac"] == pytest.approx(out["achieved"] / 6500.0)
    assert out["kernel"] == "head_fp4_kernel"


def test_roofline_e4m3_doubles_the_tensor_peak():
    cfg = CONFIGS["loop_e4m3_v262144_d2816"]
    flops, byts = bench.algorithmic(cfg)
    r = {"head_ms": [0.150], "flops": flops, "bytes": byts}
    out = bench.roofline(cfg, r, PEAKS, "measured", step_s=160e-6)
    assert out["tensor_frac_sustained"] == pytest.approx(flops / 150e-6 / 2.7e15)
    assert out["tensor_frac_burst"] == pytest.approx(flops / 150e-6 / 3.4e15)


def test_loop_breakdown_from_a_timeline():
    def t(a, b):
        return (a, b)
    tl = [{"denoise": t(0.0, 2.0), "head": t(3.0, 13.0), "merge": t(14.0, 20.0)},
          {"denoise": t(24.0, 26.0), "head": t(27.0, 37.0), "merge": t(38.0, 44.0)}]
    out = bench.loop_breakdown(tl, 2)
    assert out["denoise"] == 2.0 and out["head"] == 10.0 and out["merge"] == 6.0
    assert out["gap_denoise_head"] == 1.0 and out["gap_head_merge"] == 1.0
    assert out["gap_next_pass"] == 4.0
    assert out["per_pass"] == 22.0
    assert not math.isnan(out["per_pass"])
