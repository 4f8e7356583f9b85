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


def test_roofline_short_region_uses_the_burst_peak_and_is_hbm_bound():
    """A 20-pass run (5 ms timed region at the maximum clock) is a kernel timed alone: the burst
    tensor peak applies, so the bf16 pass is HBM-bound (t_mem 227 us > t_flop 222 us) and its
    fraction is achieved GB/s over the copy bandwidth."""
    cfg = CONFIGS["pass_bf16_v262144_d2816"]
    flops, byts = bench.algorithmic(cfg)
    clocks = {"sm_mhz": 2032.0, "sm_max_mhz": 2032.0, "reasons": []}
    regime = bench.tensor_regime(0.0054, clocks)
    assert regime == "burst"
    head_us = 263.3
    r = {"head_ms": [head_us / 1e3] * 10, "flops": flops, "bytes": byts}
    out = bench.roofline(cfg, r, PEAKS, "measured", step_s=270e-6, regime=regime)
    assert out["bound"] == "hbm" and out["unit"] == "GB/s" and out["regime"] == "burst"
    assert out["achieved"] == pytest.approx(byts / (head_us * 1e-6) / 1e9)
    assert out["frac"] == pytest.approx(out["achieved"] / 6500.0) and out["frac"] < 1.0
    assert out["t_roof_us"] == pytest.approx(byts / 6.5e12 * 1e6)
    assert out["roof_frac"] == pytest.approx(out["frac"])
    assert out["kernel_launches_timed"] == 10
    # datasheet roofline: max(bytes / 8 TB/s, flops / 2.25 PF/s) = the HBM term (184.7 us)
    assert out["datasheet_roof_frac"] == pytest.approx(byts / 8e12 / (head_us * 1e-6))
    assert out["kernel"] == "head_tc2_kernel<0>"


def test_tensor_regime_rule():
    cap = ["sw_power_cap"]
    # a seconds-long region with the power cap holding the clock down: the sustained rate
    assert bench.tensor_regime(2.0, {"sm_mhz": 1160.0, "sm_max_mhz": 2032.0, "reasons": cap}) == "sustained"
    # shorter than a second: burst, whatever the clock
    assert bench.tensor_regime(0.69, {"sm_mhz": 1140.0, "sm_max_mhz": 2032.0, "reasons": cap}) == "burst"
    assert bench.tensor_regime(0.005, {"sm_mhz": 2032.0, "sm_max_mhz": 2032.0, "reasons": []}) == "burst"
    # the clock at its maximum (power cap flagged or not): burst
    assert bench.tensor_regime(2.0, {"sm_mhz": 2032.0, "sm_max_mhz": 2032.0, "reasons": cap}) == "burst"
    # no clock samples: decided by the region's length
    assert bench.tensor_regime(2.0, {"sm_mhz": None, "sm_max_mhz": None}) == "sustained"
    assert bench.tensor_regime(0.3, {"sm_mhz": None, "sm_max_mhz": None}) == "burst"


def test_roofline_never_uses_a_sustained_peak_the_kernel_beats():
    """8 canvases at 2,109 us: 1,434 TFLOP/s, above the 1,350 sustained figure -> the burst peak."""
    cfg = CONFIGS["pass_bf16_b8_v262144_d2816"]
    flops, byts = bench.algorithmic(cfg)
    r = {"head_ms": [2.1093], "flops": flops, "bytes": byts}
    out = bench.roofline(cfg, r, PEAKS, "measured", step_s=2.11e-3, regime="sustained")
    assert out["regime"] == "burst" and out["bound"] == "tensor" and out["peak"] == 1700.0
    assert out["frac"] == pytest.approx(flops / 2.1093e-3 / 1e12 / 1700.0) and out["frac"] < 1.0


def test_roofline_sustained_regime_compute_bound_bf16():
    cfg = CONFIGS["pass_bf16_v262144_d2816"]
    flops, byts = bench.algorithmic(cfg)
    head_us = 340.0
    r = {"head_ms": [head_us / 1e3] * 4, "flops": flops, "bytes": byts}
    out = bench.roofline(cfg, r, PEAKS, "measured", step_s=350e-6, regime="sustained")
    # t_flop = 3.78e11 / 1.35e15 = 280 us > t_mem = 1.478e9 / 6.5e12 = 227 us: tensor-bound
    assert out["bound"] == "tensor" and out["unit"] == "TFLOP/s"
    assert out["achieved"] == pytest.approx(flops / (head_us * 1e-6) / 1e12)
    assert out["peak"] == 1350.0
    assert out["frac"] == pytest.approx(out["achieved"] / 1350.0) and out["frac"] < 1.0
    assert out["t_roof_us"] == pytest.approx(flops / 1.35e15 * 1e6)
    assert out["hbm_frac"] == pytest.approx(byts / (head_us * 1e-6) / 6.5e12)
    assert out["step_roof_frac"] == pytest.approx(flops / 1.35e15 / 350e-6)


def test_roofline_memory_bound_nvfp4_uses_the_hbm_peak():
    cfg = CONFIGS["pass_nvfp4_v262144_d2816"]
    flops, byts = bench.algorithmic(cfg)
    r = {"head_ms": [0.1175], "flops": flops, "bytes": byts}
    out = bench.roofline(cfg, r, PEAKS, "measured", step_s=130e-6)
    # t_flop at 6 x 1.7 PF/s = 37 us < t_mem = 64 us: HBM-bound
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


def test_roofline_fp32_head_is_bounded_by_the_cuda_cores():
    cfg = CONFIGS["pass_f32_v4096_d64"]
    flops, byts = bench.algorithmic(cfg)
    r = {"head_ms": [0.020], "flops": flops, "bytes": byts}
    out = bench.roofline(cfg, r, PEAKS, "measured", step_s=25e-6)
    alu = 148 * 128 * 2 * 2.032e9 / 1e12
    # t_flop = 1.34e8 / 77 TF/s = 1.7 us > t_mem = 1.05 MB / 6.5 TB/s = 0.16 us
    assert out["bound"] == "alu" and out["peak"] == pytest.approx(alu)
    assert out["frac"] == pytest.approx(flops / 20e-6 / 1e12 / alu)


def test_clock_summary_window_and_bracketing():
    clk = bench.ClockSampler(0)
    # (t, sm_mhz, sm_max_mhz, reasons mask, power W): power cap (0x4) active at t=1.0
    clk.rows = [(0.0, 2032, 2032, 0, 300.0), (1.0, 1200, 2032, 0x4, 1100.0),
                (1.5, 1180, 2032, 0x4, 1100.0), (3.0, 2032, 2032, 0, 250.0)]
    s = clk.summary(0.9, 1.6)
    assert s["sm_mhz"] == 1190 and s["samples"] == 2 and s["reasons"] == ["sw_power_cap"]
    assert s["window"] == "timed region"
    # a window shorter than the sampling period: the samples bracketing it
    s = clk.summary(2.0, 2.1)
    assert s["samples"] == 2 and s["sm_mhz"] == (1180 + 2032) / 2
    assert s["window"].startswith("timed region and")


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


def test_e4m3_roofline_uses_the_measured_e4m3_peak_when_there_is_one():
    """With an E4M3 GEMM rate measured in the run, the FP8 head's tensor term uses it (burst
    regime) instead of twice the bf16 rate; a measured rate below 2 x bf16 can make the head
    tensor-bound where the nominal ratio had it HBM-bound."""
    cfg = CONFIGS["loop_e4m3_v262144_d2816"]
    flops, byts = bench.algorithmic(cfg)
    r = {"head_ms": [0.150], "flops": flops, "bytes": byts}
    nominal = bench.roofline(cfg, r, PEAKS, "measured", step_s=160e-6)
    measured = bench.roofline(cfg, r, {**PEAKS, "e4m3_tflops": 3000.0}, "measured", step_s=160e-6)
    # t_flop = 3.78e11 / 3.0e15 = 126 us > t_mem = 0.74e9 / 6.5e12 = 114 us: tensor-bound
    assert measured["bound"] == "tensor" and measured["peak"] == 3000.0
    assert measured["frac"] == pytest.approx(flops / 150e-6 / 3.0e15)
    assert "measured in this run" in measured["peak_source"]
    assert measured["tensor_frac_e4m3_measured"] == pytest.approx(flops / 150e-6 / 3.0e15)
    assert nominal["bound"] == "hbm"
    # the sustained regime keeps the nominal ratio (no sustained E4M3 measurement)
    sus = bench.roofline(cfg, r, {**PEAKS, "e4m3_tflops": 3000.0}, "measured", step_s=160e-6,
                         regime="sustained")
    assert "x2 nominal" in sus.get("peak_source", "") or sus["bound"] == "hbm"
