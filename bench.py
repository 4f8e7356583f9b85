"""Benchmark of the canvas pass on B300: canvas passes/s (and slots/s) and % of roofline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

One step = one pass of the whole hot path over one batch of synthetic inputs: the vocabulary
head contraction with fused softmax statistics, the cross-group merge, the confidence top-K
keep, the counter-hash re-randomisation and the stop test (dg_canvas_step with a device stop
state). Loop configurations time one full dg_canvas_loop per step and count the passes it ran.
The default workload is one 256-slot canvas over a 262144-token bf16 head with d = 2816.

Under torchrun (N > 1) every rank runs an independent replica on its own GPU (the path has no
exchange step); the timed region is bracketed by barriers and the max over ranks is reported.
Prints ONE JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_CONFIG = "pass_bf16_v262144_d2816"
L2_BYTES = 126 * 1024 * 1024


# ---------------------------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ---------------------------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws: int, backend: str):
    if ws > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend=backend)


def barrier(ws: int):
    if ws > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, ws: int, device) -> float:
    if ws == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate(units_per_rank: float, seconds_max: float, ws: int) -> float:
    """Whole-job throughput: the units every rank processed over the slowest rank's time."""
    return units_per_rank * ws / seconds_max


# ---------------------------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------------------------
# NVML clock-event reason bits (nvmlClocksEventReason*)
REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
               "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80}


class Nvml:
    """The few read-only NVML queries the clock sampler needs, through ctypes on the driver's
    libnvidia-ml.so.1 (no Python NVML package is required)."""
    CLOCK_SM = 1

    def __init__(self, dev_index: int):
        import ctypes as C
        self.C = C
        self.lib = C.CDLL("libnvidia-ml.so.1")
        init = getattr(self.lib, "nvmlInit_v2", None) or self.lib.nvmlInit
        self._ok(init())
        self.h = C.c_void_p()
        props = torch.cuda.get_device_properties(dev_index)
        rc = self.lib.nvmlDeviceGetHandleByUUID(("GPU-" + str(props.uuid)).encode(),
                                                C.byref(self.h))
        if rc != 0:
            bus = f"{props.pci_domain_id:08X}:{props.pci_bus_id:02X}:{props.pci_device_id:02X}.0"
            f = getattr(self.lib, "nvmlDeviceGetHandleByPciBusId_v2", None) or \
                self.lib.nvmlDeviceGetHandleByPciBusId
            self._ok(f(bus.encode(), C.byref(self.h)))
        self._reasons = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    @staticmethod
    def _ok(rc):
        if rc != 0:
            raise RuntimeError(f"NVML error {rc}")

    def max_sm_mhz(self) -> int:
        v = self.C.c_uint()
        self._ok(self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.CLOCK_SM, self.C.byref(v)))
        return v.value

    def sample(self, mx: int):
        C = self.C
        sm, rs, mw = C.c_uint(), C.c_ulonglong(), C.c_uint()
        self._ok(self.lib.nvmlDeviceGetClockInfo(self.h, self.CLOCK_SM, C.byref(sm)))
        self._ok(self._reasons(self.h, C.byref(rs)))
        self._ok(self.lib.nvmlDeviceGetPowerUsage(self.h, C.byref(mw)))
        return (time.perf_counter(), sm.value, mx, rs.value, mw.value / 1e3)


class ClockSampler:
    """Samples the SM clock, its maximum, the clock-event reasons and the power draw every
    `period_s` from a background thread with read-only NVML queries (Nvml), for the whole life of the
    `with` block (warm-up, timed and end-to-end legs), so that even a timed region of a few
    milliseconds has samples around it. mark() stamps host times; summary(t0, t1) reports the
    samples taken between two stamps (or, if the window is shorter than the sampling period,
    the samples that bracket it)."""

    def __init__(self, dev_index: int, period_s: float = 0.002):
        self.dev_index = dev_index
        self.period = period_s
        self.rows = []          # (t, sm_mhz, sm_max_mhz, reasons_mask, power_w)
        self.error = None
        self._stop = None

    def __enter__(self):
        import threading
        try:
            nv = Nvml(self.dev_index)
            mx = nv.max_sm_mhz()
            self.rows.append(nv.sample(mx))
        except Exception as e:     # no NVML: report why instead of clocks
            self.error = f"NVML unavailable: {e!r}"[:200]
            return self
        self._stop = threading.Event()

        def poll():
            while not self._stop.is_set():
                try:
                    self.rows.append(nv.sample(mx))
                except Exception as e:
                    self.error = repr(e)[:200]
                    return
                self._stop.wait(self.period)

        self._thread = threading.Thread(target=poll, daemon=True)
        self._thread.start()
        return self

    def __exit__(self, *a):
        if self._stop is not None:
            self._stop.set()
            self._thread.join(timeout=5)

    @staticmethod
    def mark() -> float:
        return time.perf_counter()

    def summary(self, t0: float, t1: float) -> dict:
        if self.error and not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [self.error]}
        rows = [r for r in self.rows if t0 <= r[0] <= t1]
        window = "timed region"
        if len(rows) < 2:
            before = [r for r in self.rows if r[0] < t0][-1:]
            after = [r for r in self.rows if r[0] > t1][:1]
            rows = before + rows + after
            window = "timed region and the samples bracketing it"
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        reasons = sorted({n for r in rows for n, bit in REASON_BITS.items() if r[3] & bit})
        return {"sm_mhz": statistics.median(r[1] for r in rows),
                "sm_max_mhz": max(r[2] for r in rows), "reasons": reasons,
                "samples": len(rows), "window": window, "source": "nvml",
                "power_w_max": round(max(r[4] for r in rows), 1)}


# ---------------------------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------------------------
def to_dev_bf16(bits, shape):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).reshape(shape).cuda()


def algorithmic(cfg):
    """FLOPs and algorithmic bytes of one pass (operands read once, O(R) outputs)."""
    flops = 2.0 * cfg.R * cfg.V * cfg.d
    out_bytes = cfg.R * (4 + 4 + 4 + 1 + 4)
    if cfg.precision == "nvfp4":
        # W codes (4 bits) + E4M3 block scales (1 per 16) + fp32 row scales; bf16 h in
        return flops, cfg.V * cfg.d / 2 + cfg.V * cfg.d / 16 + cfg.V * 4 + cfg.R * cfg.d * 2 + out_bytes
    eb = {"f32": 4, "bf16": 2, "e4m3": 1}[cfg.precision]
    byts = cfg.V * cfg.d * eb + cfg.R * cfg.d * eb + out_bytes
    if cfg.precision == "e4m3":
        byts += cfg.V * 4 + cfg.R * 4
    return flops, byts


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}, "fallback"


DATASHEET = {"hbm_gbs": 8000.0, "bf16_tflops": 2250.0, "e4m3_tflops": 4500.0}


def measure_e4m3_peak(device, n=8192, reps=10):
    """Dense E4M3 tensor rate of this GPU, measured the way the bf16 peak is: a cuBLAS GEMM
    (torch._scaled_mm, E4M3 x E4M3 -> bf16, n^3, unit scales), 3 untimed and `reps` timed calls
    between CUDA events, as a burst. None if the library call is unavailable."""
    try:
        g = torch.Generator(device=device).manual_seed(0)
        a = torch.randn(n, n, device=device, generator=g).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device=device, generator=g).to(torch.float8_e4m3fn)
        one = torch.ones((), device=device, dtype=torch.float32)
        mm = lambda: torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        for _ in range(3):
            mm()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            mm()
        e1.record()
        torch.cuda.synchronize()
        s = e0.elapsed_time(e1) / 1e3 / reps
        del a, b
        torch.cuda.empty_cache()
        return 2.0 * n ** 3 / s / 1e12
    except (RuntimeError, AttributeError, TypeError):
        return None

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of the head kernel,
# from an ncu capture of the build whose head sources hash to `src` (summaries in profiles/).
# A different hash means the kernel changed since the counters were taken: traffic is null.
HEAD_SOURCES = {
    "tc2": ["dg_head_tc2.cu", "dg_head_epi.cuh", "dg_common.cuh", "dg_ptx.cuh", "dg_internal.h"],
    "fp4": ["dg_head_fp4.cu", "dg_head_epi.cuh", "dg_common.cuh", "dg_ptx.cuh", "dg_internal.h"],
}
TRAFFIC = {
    "pass_bf16_v262144_d2816": {"bytes": 1.477882752e9 + 1.546624e6, "src": "c118b87f934b035b"},
    "loop_e4m3_v262144_d2816": {"bytes": 740.019712e6 + 1.556864e6, "src": "c118b87f934b035b"},
    "pass_nvfp4_v262144_d2816": {"bytes": 417.154944e6 + 2.19584e6, "src": "5a2dd153528e1ca7"},
}


def head_source_hash(kind: str = "tc2") -> str:
    import hashlib
    hsh = hashlib.sha256()
    for f in HEAD_SOURCES[kind]:
        with open(os.path.join(ROOT, "uniform_state_denoising_vocab_b300", "csrc", f), "rb") as fh:
            hsh.update(fh.read())
    return hsh.hexdigest()[:16]


SUSTAINED_MIN_S = 1.0    # a timed region at least this long runs at the power-capped clock
NEAR_MAX_CLOCK = 0.95    # a median SM clock within 5% of its maximum is an unthrottled run
ALU_FP32_FLOP_PER_CLK = 148 * 128 * 2   # fp32 FMA lanes x 2 flops, for the CUDA-core head


def tensor_regime(timed_s: float, clocks: dict) -> str:
    """Which measured tensor peak applies to a kernel timed inside a region of `timed_s`
    seconds: the sustained (power-capped) rate for a region of a second or more during which the
    sampled clocks show the power cap holding the SM clock below 95% of its maximum (or, with no
    clock samples, for any region of a second or more); the burst rate otherwise."""
    sm, mx = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    if timed_s < SUSTAINED_MIN_S:
        return "burst"
    if sm is None or not mx:
        return "sustained"
    capped = "sw_power_cap" in clocks.get("reasons", []) and sm < NEAR_MAX_CLOCK * mx
    return "sustained" if capped else "burst"


def roofline(cfg, r, peaks, peak_kind, step_s, regime="burst"):
    """Roofline of the head kernel (the dominant kernel): t_roof = max(FLOPs / tensor peak,
    algorithmic bytes / HBM bandwidth), `bound` the slower term, frac = t_roof / kernel time
    (= achieved / peak of the bound). The HBM peak is the measured copy bandwidth; the tensor
    peak is the measured bf16 cuBLAS rate of the timed region's regime (burst or sustained, see
    tensor_regime), x2 for E4M3 and x6 for NVFP4 (the nominal dense ratios 4.5 and 13.5 to
    2.25 PFLOP/s). The fp32 head runs on the CUDA cores: its compute peak is 148 SMs x 128 FMA
    lanes x 2 flops at the maximum SM clock (2,032 MHz), bound "alu". The datasheet roofline
    (8 TB/s, 2.25 PFLOP/s dense bf16) is reported beside it."""
    head_s = statistics.mean(r["head_ms"]) / 1e3
    ratio = {"e4m3": 2.0, "nvfp4": 6.0}.get(cfg.precision, 1.0)
    e4m3_measured = peaks.get("e4m3_tflops") if cfg.precision == "e4m3" else None
    if regime == "sustained" and cfg.precision != "f32":
        sus = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) * ratio * 1e12
        if r["flops"] / head_s > sus:   # a rate the kernel beats is no ceiling: use the burst one
            regime = "burst"
    bf16 = peaks["bf16_tflops"] if regime == "burst" else peaks.get("bf16_tflops_sustained",
                                                                     peaks["bf16_tflops"])
    if cfg.precision == "f32":
        tens, tunit = ALU_FP32_FLOP_PER_CLK * 2.032e9 / 1e12, "alu"
        src = "fp32 FMA lanes x maximum SM clock"
    elif e4m3_measured and regime == "burst":
        tens, tunit = e4m3_measured, "tensor"
        src = "E4M3 cuBLAS (torch._scaled_mm 8192^3) measured in this run, burst"
    else:
        tens, tunit = bf16 * ratio, "tensor"
        src = f"{peak_kind} {regime} bf16 cuBLAS" + \
            (f" x{ratio:g} nominal {cfg.precision}/bf16" if ratio != 1.0 else "")
    t_mem = r["bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_flop = r["flops"] / (tens * 1e12)
    out = {}
    if t_mem >= t_flop:
        achieved = r["bytes"] / head_s / 1e9
        out.update(bound="hbm", achieved=achieved, peak=peaks["hbm_gbs"], unit="GB/s",
                   frac=achieved / peaks["hbm_gbs"], peak_source=f"{peak_kind} copy bandwidth")
    else:
        achieved = r["flops"] / head_s / 1e12
        out.update(bound=tunit, achieved=achieved, peak=tens, unit="TFLOP/s",
                   frac=achieved / tens, peak_source=src)
    out["regime"] = regime
    rec = TRAFFIC.get(cfg.name)
    kind = "fp4" if cfg.precision == "nvfp4" else "tc2"
    out["traffic"] = rec["bytes"] if rec and rec["src"] == head_source_hash(kind) else None
    out["kernel"] = ("head_fp4_kernel" if cfg.precision == "nvfp4" else
                     {"f32": "head_simt_kernel", "bf16": "head_tc2_kernel<0>",
                      "e4m3": "head_tc2_kernel<1>"}[cfg.precision] if cfg.R > 128 or cfg.precision == "f32"
                     else {"bf16": "head_tc_kernel<0>", "e4m3": "head_tc_kernel<1>"}[cfg.precision])
    out["kernel_us"] = head_s * 1e6
    out["kernel_launches_timed"] = len(r["head_ms"])
    if r.get("head_clock"):
        out["kernel_sm_mhz_effective"] = r["head_clock"]["sm_mhz_effective"]
        out["kernel_kcycles"] = r["head_clock"]["head_kcycles"]
    out["t_roof_us"] = max(t_mem, t_flop) * 1e6
    out["roof_frac"] = max(t_mem, t_flop) / head_s
    out["hbm_frac"] = r["bytes"] / head_s / 1e9 / peaks["hbm_gbs"]
    if cfg.precision != "f32":
        out["tensor_frac_burst"] = r["flops"] / head_s / 1e12 / (peaks["bf16_tflops"] * ratio)
        out["tensor_frac_sustained"] = r["flops"] / head_s / 1e12 / (
            peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) * ratio)
        if e4m3_measured:
            out["tensor_frac_e4m3_measured"] = r["flops"] / head_s / 1e12 / e4m3_measured
        ds_t = max(r["bytes"] / (DATASHEET["hbm_gbs"] * 1e9),
                   r["flops"] / (DATASHEET["bf16_tflops"] * ratio * 1e12))
        out["datasheet_t_roof_us"] = ds_t * 1e6
        out["datasheet_roof_frac"] = ds_t / head_s
        out["datasheet_step_roof_frac"] = ds_t / step_s
    out["step_roof_frac"] = max(t_mem, t_flop) / step_s
    return out


def loop_breakdown(tl, passes):
    """Mean per-pass durations (us) of the loop's kernels and the gaps between them, from the
    per-pass kernel timeline: denoise, head, merge, and the gaps denoise->head, head->merge and
    merge->next pass's denoise (the graph's conditional iteration)."""
    keys = ("denoise", "gap_denoise_head", "head", "gap_head_merge", "merge", "gap_next_pass")
    acc = {k: [] for k in keys}
    for p in range(passes):
        d, h, m = tl[p]["denoise"], tl[p]["head"], tl[p]["merge"]
        if d is None or h is None or m is None:
            continue
        acc["denoise"].append(d[1] - d[0])
        acc["gap_denoise_head"].append(h[0] - d[1])
        acc["head"].append(h[1] - h[0])
        acc["gap_head_merge"].append(m[0] - h[1])
        acc["merge"].append(m[1] - m[0])
        if p + 1 < passes and tl[p + 1]["denoise"] is not None:
            acc["gap_next_pass"].append(tl[p + 1]["denoise"][0] - m[1])
    out = {k: (round(statistics.mean(v), 2) if v else None) for k, v in acc.items()}
    if passes > 1 and tl[0]["denoise"] is not None and tl[passes - 1]["merge"] is not None:
        out["per_pass"] = round((tl[passes - 1]["merge"][1] - tl[0]["denoise"][0]) / passes, 2)
    return out




def _launch_checked(rc, dg):
    if rc != 0:
        raise RuntimeError(dg.dg_status_string(rc))


def pass_inputs(cfg, dg, dev):
    """Device inputs of a single-pass workload. The NVFP4 head is generated in bf16 and quantised
    on the device by the library's own quantiser (dg_quantize_nvfp4): the same operand format a
    4-bit checkpoint stores, without the slow host quantisation the parity tests use."""
    import dataclasses
    from workloads import make_pass_inputs
    R, d, V = cfg.R, cfg.d, cfg.V
    src = dataclasses.replace(cfg, precision="bf16") if cfg.precision == "nvfp4" else cfg
    x = make_pass_inputs(src)
    dkw = {}
    if cfg.precision == "f32":
        h = torch.from_numpy(x["h"]).view(R, d).cuda()
        w = torch.from_numpy(x["w"]).view(V, d).cuda()
        wsc = None
    elif cfg.precision == "nvfp4":
        h = to_dev_bf16(x["h"], (R, d))
        wq = dg.dg_quantize_nvfp4(to_dev_bf16(x["w"], (V, d)))
        w, wsc = wq["codes"], wq["scale"]
        dkw = dict(w_dtype=dg.DG_NVFP4, w_block_scale=wq["block_scale"])
    elif cfg.precision == "bf16":
        h, w, wsc = to_dev_bf16(x["h"], (R, d)), to_dev_bf16(x["w"], (V, d)), None
    else:
        h = to_dev_bf16(x["h"], (R, d))
        w = torch.from_numpy(x["w"]).view(V, d).cuda()
        wsc = torch.from_numpy(x["w_scale"]).cuda()
    canvas = torch.from_numpy(x["canvas"]).cuda()
    torch.cuda.synchronize()
    return h, w, wsc, dkw, canvas


def run_pass(cfg, steps, warmup, ws_, clk, e2e_steps=0):
    """`steps` back-to-back canvas passes (dg_canvas_step with a device stop state whose rule
    never fires) timed with CUDA events on the launching stream; the head kernel of every
    HEAD_SAMPLE-th pass is bracketed by its own events. Then, if e2e_steps, the end-to-end leg
    through dg_canvas_step_host on page-locked host buffers."""
    import ctypes as C
    import uniform_state_denoising_vocab_b300 as dg
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    flops, byts = algorithmic(cfg)
    R = cfg.R
    launches_per_step = 2 + (1 if cfg.precision in ("e4m3", "nvfp4") else 0)
    h, w, wsc, dkw, canvas = pass_inputs(cfg, dg, dev)
    canvas_out = torch.empty_like(canvas)
    state = dg.new_state(cfg.B, dev)
    rule = dg.StopRule(max_passes=1 << 30, entropy_threshold=0.0, stable_passes=1 << 30,
                       stop_mode=dg.STOP_OR)
    desc = dg.make_desc(h, w, B=cfg.B, S=cfg.S, w_scale=wsc, **dkw)
    wsb = torch.empty(dg.dg_workspace_bytes(desc) + 256, dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    outs = {"argmax": torch.empty(R, dtype=torch.int32, device=dev),
            "conf": torch.empty(R, device=dev), "entropy": torch.empty(R, device=dev),
            "kept": torch.empty(R, dtype=torch.uint8, device=dev),
            "mean_entropy": torch.empty(cfg.B, device=dev)}
    L = dg.lib()
    P = lambda t: C.c_void_p(t.data_ptr()) if t is not None else None
    sh = C.c_void_p(stream.cuda_stream)
    rref, dref = C.byref(rule), C.byref(desc)

    def step(i, cin, cout):
        _launch_checked(L.dg_canvas_step(dref, P(cin), P(cout), cfg.keep_k, C.c_uint64(cfg.seed),
                                         C.c_uint32(i), P(outs["argmax"]), P(outs["conf"]),
                                         P(outs["entropy"]), P(outs["kept"]),
                                         P(outs["mean_entropy"]), P(state), rref, P(wsb),
                                         wsb.numel(), P(status), sh), dg)

    for i in range(warmup):
        step(i, canvas, canvas_out)
    torch.cuda.synchronize()
    # The head kernel of every HEAD_SAMPLE-th pass is bracketed by events on the launching
    # stream (at least 8 launches whatever the step count, when there are 8 steps): an event
    # pair between the kernels of a pass breaks their programmatic dependent launch, so
    # bracketing every pass would slow the passes being timed.
    sample = max(1, min(8, steps // 8))
    heads = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(0, steps, sample)]
    # each bracketed head also writes its SM clock sample (clock64 and global timer in CTA 0)
    clk_samples = torch.zeros(len(heads), 4, dtype=torch.int64, device=dev)
    for a_, b_ in heads:    # create the event handles outside the timed region
        a_.record(stream)
        b_.record(stream)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws_)
    torch.cuda.synchronize()
    t0 = clk.mark()
    ev0.record(stream)
    for i in range(steps):
        if i % sample == sample - 1:
            dg.dg_profile_next_head(*heads[i // sample])
            dg.dg_profile_next_head_clock(clk_samples[i // sample])
        step(warmup + i, canvas if i % 2 == 0 else canvas_out, canvas_out if i % 2 == 0 else canvas)
    ev1.record(stream)
    torch.cuda.synchronize()
    t1 = clk.mark()
    barrier(ws_)
    t_ms = ev0.elapsed_time(ev1)
    head_ms = [a.elapsed_time(b) for a, b in heads[: steps // sample]]
    out = {"t_s": t_ms / 1e3, "units": cfg.B * steps, "head_ms": head_ms,
           "head_clock": dg.sm_clock_stats(clk_samples[: steps // sample]),
           "clocks": clk.summary(t0, t1), "status": int(status.item()),
           "launches": launches_per_step * steps, "flops": flops, "bytes": byts}
    if e2e_steps:
        # end to end through the host-buffer entry point (dg_canvas_step_host): every step
        # uploads its hidden states and canvas from page-locked host memory and reads its new
        # canvas and mean entropy back, inside the timed region. The library alternates two
        # staging sets in its workspace, so a step's uploads overlap the previous step's kernels.
        h_host = h.cpu().pin_memory()
        c_host = canvas.cpu().pin_memory()
        c_back = torch.empty_like(c_host).pin_memory()
        m_back = torch.empty(cfg.B, dtype=torch.float32).pin_memory()
        hdesc = dg.host_desc(h_host, w, B=cfg.B, S=cfg.S, w_scale=wsc, **dkw)
        wsh = torch.empty(dg.dg_workspace_bytes_host(hdesc), dtype=torch.uint8, device=dev)
        hdref = C.byref(hdesc)

        def e2e_step(i):
            _launch_checked(L.dg_canvas_step_host(hdref, P(c_host), P(c_back), P(m_back),
                                                  cfg.keep_k, C.c_uint64(cfg.seed), C.c_uint32(i),
                                                  P(state), rref, P(wsh), wsh.numel(), P(status),
                                                  sh), dg)

        e2e_step(0)                         # first call creates the library's copy stream
        barrier(ws_)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(e2e_steps):
            e2e_step(i)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(ws_)
        out.update(e2e_t_s=e0.elapsed_time(e1) / 1e3, e2e_units=cfg.B * e2e_steps,
                   h2d=h_host.numel() * h_host.element_size() + c_host.numel() * 4,
                   d2h=c_back.numel() * 4 + m_back.numel() * 4)
    return out


def run_loop(cfg, steps, warmup, ws_, clk, e2e_steps=0):
    """`steps` whole loops (one dg_canvas_loop each: denoiser, quantiser, head and merge per
    pass, until the stop rule) timed with CUDA events; the passes they ran are the units. The
    head alone is timed with events around standalone launches on the loop's last hidden states
    (kernels inside the loop's graph cannot be bracketed), and the in-graph per-pass breakdown
    comes from the library's kernel timeline on one more (untimed) loop."""
    import ctypes as C
    import uniform_state_denoising_vocab_b300 as dg
    from workloads import make_loop_inputs
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    flops, byts = algorithmic(cfg)
    R, d, V = cfg.R, cfg.d, cfg.V
    x = make_loop_inputs(cfg)
    if cfg.precision == "bf16":
        w, wsc = to_dev_bf16(x["w"], (V, d)), None
    else:
        w = torch.from_numpy(x["w"]).view(V, d).cuda()
        wsc = torch.from_numpy(x["w_scale"]).cuda()
    y = torch.from_numpy(x["y"]).cuda()
    del x
    canvas = torch.empty(R, dtype=torch.int32, device=dev)
    hbuf = torch.empty(R, d, dtype=torch.bfloat16, device=dev)
    state = dg.new_state(cfg.B, dev)
    desc = dg.make_desc(hbuf, w, B=cfg.B, S=cfg.S, w_scale=wsc)
    wsb = torch.empty(dg.dg_workspace_bytes(desc) + 256, dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    loop_out = {"argmax": torch.empty(R, dtype=torch.int32, device=dev),
                "conf": torch.empty(R, device=dev), "entropy": torch.empty(R, device=dev)}
    kw = dict(B=cfg.B, S=cfg.S, theta=cfg.theta, y=y, h_buffer=hbuf, w_scale=wsc,
              keep_k0=cfg.keep_k, seed=cfg.seed, max_passes=cfg.max_passes,
              stable_passes=cfg.stable_passes, n_content=cfg.n_content, s_content=cfg.s_content,
              s_pad=cfg.s_pad, state=state, workspace=wsb, status=status, outputs=loop_out)
    # the call's arguments are marshalled once; each step issues the C call (one graph launch)
    loop = dg.prepare_loop(w, canvas, **kw)
    for _ in range(warmup):
        loop.run()
    torch.cuda.synchronize()
    passes_per_loop = int(dg.state_fields(state)["passes"].sum())
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws_)
    torch.cuda.synchronize()
    t0 = clk.mark()
    ev0.record(stream)
    for _ in range(steps):
        loop.run()
    ev1.record(stream)
    torch.cuda.synchronize()
    t1 = clk.mark()
    barrier(ws_)
    t_ms = ev0.elapsed_time(ev1)
    out = {"t_s": t_ms / 1e3, "units": passes_per_loop * steps, "clocks": clk.summary(t0, t1),
           "status": int(status.item()), "flops": flops, "bytes": byts,
           "passes_per_loop": passes_per_loop,
           "launches": steps * (1 + (3 + (1 if cfg.precision == "e4m3" else 0)) * passes_per_loop)}
    if e2e_steps:
        # end to end: targets in, final canvas + state out, every loop
        y_host = y.cpu().pin_memory()
        c_back = torch.empty(R, dtype=torch.int32).pin_memory()
        s_back = torch.empty_like(state, device="cpu").pin_memory()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            y.copy_(y_host, non_blocking=True)
            loop.run()
            c_back.copy_(canvas, non_blocking=True)
            s_back.copy_(state, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        out.update(e2e_t_s=e0.elapsed_time(e1) / 1e3, e2e_units=passes_per_loop * e2e_steps,
                   h2d=y_host.numel() * 4, d2h=c_back.numel() * 4 + s_back.numel() * 4)
    # the dominant kernel alone: the head over the loop's last hidden states
    L = dg.lib()
    P = lambda t: C.c_void_p(t.data_ptr()) if t is not None else None
    sa = torch.empty(R, dtype=torch.int32, device=dev)
    sc, se = torch.empty(R, device=dev), torch.empty(R, device=dev)
    sm = torch.empty(cfg.B, device=dev)
    heads = []
    n_head = max(20, min(400, steps * passes_per_loop))
    clk_samples = torch.zeros(n_head, 4, dtype=torch.int64, device=dev)
    for i in range(n_head):
        ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        dg.dg_profile_next_head(*ev)
        dg.dg_profile_next_head_clock(clk_samples[i])
        _launch_checked(L.dg_canvas_stats(C.byref(desc), P(sa), P(sc), P(se), P(sm), P(wsb),
                                          wsb.numel(), P(status),
                                          C.c_void_p(stream.cuda_stream)), dg)
        heads.append(ev)
    torch.cuda.synchronize()
    out["head_ms"] = [a.elapsed_time(b) for a, b in heads[len(heads) // 4:]]
    out["head_clock"] = dg.sm_clock_stats(clk_samples[len(heads) // 4:])
    # in-graph breakdown of one more (untimed) loop from the library's per-pass kernel timeline,
    # with each pass's head clock sample (effective SM clock, head cycles)
    rt = dg.dg_canvas_loop(w, canvas, timeline=True, sm_clock=True, **kw)
    torch.cuda.synchronize()
    npass = int(dg.state_fields(rt["state"])["passes"].max())
    out["loop_breakdown_us"] = loop_breakdown(dg.timeline_us(rt["trace_timeline"], cfg.max_passes),
                                              npass)
    hc = dg.sm_clock_stats(rt["trace_sm_clock"][:npass])
    out["loop_breakdown_us"]["head_sm_mhz_effective"] = hc["sm_mhz_effective"]
    out["loop_breakdown_us"]["head_kcycles"] = hc["head_kcycles"]
    return out


# Extra workloads measured in the same run (one GPU only), each sized so its timed region is
# a fraction of a second: (steps, warm-up).
EXTRA_WORKLOADS = {
    "pass_bf16_v262144_d2816": (500, 10),
    "loop_e4m3_v262144_d2816": (40, 3),
    "pass_bf16_b8_v262144_d2816": (150, 5),
    "pass_nvfp4_v262144_d2816": (1000, 20),
    "loop_bf16_v32768_d256": (300, 5),
    "pass_f32_v4096_d64": (2000, 20),
}


def summarise(cfg, r, peaks, peak_kind, ws_=1):
    """Throughput, roofline and clocks of one measured workload."""
    step_s = r["t_s"] / (r["units"] / cfg.B)
    rec = {"value": aggregate(r["units"], r["t_s"], ws_), "unit": "canvas passes/s",
           "slots_per_s": aggregate(r["units"], r["t_s"], ws_) * cfg.S,
           "ms_per_pass": step_s * 1e3, "timed_s": r["t_s"], "clocks": r["clocks"],
           "device_status": r["status"]}
    if r.get("head_ms"):
        rec["roofline"] = roofline(cfg, r, peaks, peak_kind, step_s,
                                   tensor_regime(r["t_s"], r["clocks"]))
    if cfg.mode == "loop":
        rec["passes_per_loop"] = r["passes_per_loop"]
        rec["loop_breakdown_us"] = r["loop_breakdown_us"]
    return rec


# ---------------------------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------------------------
class OracleSampler:
    """The oracle timed on a bounded sample of the workload: a few slot rows against the full
    vocabulary (statistics), plus the keep/re-randomise step for the whole canvas, scaled to
    one canvas pass by rows. size(target_s) sizes the sample after a calibration on one row per
    host thread (the oracle spreads rows over threads) that follows one warm-up row (thread
    start-up, first touch of W)."""

    def __init__(self, cfg):
        import oracle
        from workloads.gen import make_head, normal_f32, f32_to_bf16_bits, TAG_H
        oracle.build()
        self.o, self.cfg = oracle, cfg
        V, d, R = cfg.V, cfg.d, cfg.R
        head = make_head(cfg)
        self.w, self.wsc = head["w"], head["w_scale"]
        h = normal_f32(R * d, cfg.seed, TAG_H)
        if cfg.precision != "f32":
            h = f32_to_bf16_bits(h)
        self.hs = None
        self.bkw = {}
        if cfg.precision == "e4m3":
            h, self.hs = oracle.quant_rows_e4m3(h, R, d)
        if cfg.precision == "nvfp4":
            h, hb, self.hs = oracle.quant_rows_nvfp4(h, R, d)
            self.bkw = dict(h_bscale=hb, w_bscale=head["w_bscale"])
        self.h = h
        self.rows = 1
        self._stats(1)

    def _stats(self, rows):
        c = self.cfg
        return self.o.head_stats(c.R, c.d, c.V, c.precision, self.h, self.w, h_scale=self.hs,
                                 w_scale=self.wsc, rows=np.arange(rows), **self.bkw)

    def size(self, target_s: float):
        cal = min(max(1, self.o.num_threads()), self.cfg.R)
        t0 = time.perf_counter()
        self._stats(cal)
        t1 = (time.perf_counter() - t0) / cal
        self.rows = int(max(1, min(self.cfg.R, target_s / max(t1, 1e-6))))
        return self

    def step(self) -> float:
        """Seconds per canvas pass, estimated from one timed sample."""
        c = self.cfg
        t0 = time.perf_counter()
        st = self._stats(self.rows)
        t_stats = time.perf_counter() - t0
        idx = np.arange(c.R) % self.rows   # the per-canvas step on the full canvas
        t0 = time.perf_counter()
        self.o.select(c.B, c.S, c.V, st["argmax"][idx], st["conf"][idx], st["entropy"][idx],
                      c.keep_k, c.seed, 0)
        t_sel = time.perf_counter() - t0
        return t_stats * (c.R / self.rows) + t_sel

    def describe(self) -> str:
        c = self.cfg
        return (f"{self.rows} of {c.R} slot rows x full vocabulary {c.V} x d={c.d} (statistics), "
                f"plus the keep/re-randomise step on all {c.R} rows; scaled by rows to one pass")

    def cores(self) -> int:
        return self.o.num_threads()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workloads", default="all", choices=["all", "none"],
                    help="also measure the other full-size workloads (one GPU only)")
    args = ap.parse_args()
    from workloads import CONFIGS
    cfg = CONFIGS[args.config]
    ws_, rank, local = dist_env()
    metric = "canvas passes/s (256 slots x 262K vocab, d=2816) and % of roofline, 1 B300"
    workload = {"workload": cfg.name, "canvases": cfg.B, "slots": cfg.S, "vocab": cfg.V,
                "hidden": cfg.d, "precision": cfg.precision, "mode": cfg.mode,
                "keep_k": cfg.keep_k, "seed": cfg.seed,
                "l2": "inputs larger than L2 (head %.2f GB), no flush" % (cfg.V * cfg.d * {"f32": 4, "bf16": 2, "e4m3": 1, "nvfp4": 0.5625}[cfg.precision] / 1e9)
                if cfg.V * cfg.d > L2_BYTES else "L2-resident head, latency-bound"}

    if args.impl == "reference":
        if rank != 0:
            return
        # each step times one bounded sample, sized so that the whole run stays near 1.5 min
        smp = OracleSampler(cfg).size(min(10.0, max(0.5, 90.0 / max(1, args.steps + args.warmup))))
        for _ in range(args.warmup):
            smp.step()
        per = [smp.step() for _ in range(args.steps)]
        v = len(per) / sum(per)
        line = {"impl": "reference", "metric": metric, "value": v, "unit": "canvas passes/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": statistics.mean(per) * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": workload,
                "cpu_baseline": {"value": v, "unit": "canvas passes/s", "cores": smp.cores(),
                                 "kind": "oracle", "sample": smp.describe()},
                "e2e": {"value": v, "unit": "canvas passes/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    init_dist(ws_, "nccl")
    torch.cuda.set_device(local)
    peaks, peak_kind = load_peaks()
    run = run_pass if cfg.mode == "pass" else run_loop
    e2e_steps = max(10, args.steps // 4) if cfg.mode == "pass" else max(3, args.steps // 4)
    with ClockSampler(torch.cuda.current_device()) as clk:
        r = run(cfg, args.steps, args.warmup, ws_, clk, e2e_steps=e2e_steps)
        raw = {}
        if args.workloads == "all" and ws_ == 1:
            for name, (k, w) in EXTRA_WORKLOADS.items():
                if name == cfg.name:
                    continue
                c = CONFIGS[name]
                raw[name] = (run_pass if c.mode == "pass" else run_loop)(c, k, w, 1, clk)
                torch.cuda.empty_cache()
    # the E4M3 tensor peak, measured after every timed region so that it heats none of them
    if cfg.precision == "e4m3" or any(CONFIGS[n].precision == "e4m3" for n in raw):
        e4 = measure_e4m3_peak(torch.device("cuda", local))
        if e4:
            peaks = {**peaks, "e4m3_tflops": e4}
    extras = {name: summarise(CONFIGS[name], rr, peaks, peak_kind) for name, rr in raw.items()}
    t_max = max_over_ranks(r["t_s"], ws_, torch.device("cuda", local))
    e_max = max_over_ranks(r["e2e_t_s"], ws_, torch.device("cuda", local))
    if rank != 0:
        if ws_ > 1:
            torch.distributed.destroy_process_group()
        return
    value = aggregate(r["units"], t_max, ws_)
    e2e = aggregate(r["e2e_units"], e_max, ws_)
    line = {"metric": metric, "value": value, "unit": "canvas passes/s", "n_gpus": ws_,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_max * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": {"f32": "f32", "bf16": "bf16", "e4m3": "e4m3", "nvfp4": "nvfp4"}[cfg.precision],
            "data": "synthetic (seeded N(0,1) hidden states, N(0,1/d) head)",
            "config": workload, "slots_per_s": value * cfg.S,
            "e2e": {"value": e2e, "unit": "canvas passes/s", "h2d_bytes_per_step": r["h2d"],
                    "d2h_bytes_per_step": r["d2h"]},
            "gpu_launches": r["launches"], "clocks": r["clocks"], "device_status": r["status"],
            "peaks": {"source": peak_kind, **{k: peaks[k] for k in ("hbm_gbs", "bf16_tflops")
                                              if k in peaks},
                      "bf16_tflops_sustained": peaks.get("bf16_tflops_sustained"),
                      "e4m3_tflops": peaks.get("e4m3_tflops"),
                      "e4m3_source": ("torch._scaled_mm 8192^3, burst, measured in this run"
                                      if peaks.get("e4m3_tflops") else "2 x bf16 (nominal ratio)")}}
    if r.get("head_ms"):
        step_s = t_max / (r["units"] / cfg.B)
        line["roofline"] = roofline(cfg, r, peaks, peak_kind, step_s,
                                    tensor_regime(t_max, r["clocks"]))
        if cfg.mode == "loop":
            line["passes_per_loop"] = r["passes_per_loop"]
            line["loop_breakdown_us"] = r["loop_breakdown_us"]
    if extras:
        line["workloads"] = extras
    if not args.no_cpu_baseline and ws_ == 1:
        smp = OracleSampler(cfg).size(15.0)
        per = smp.step()
        line["cpu_baseline"] = {"value": 1.0 / per, "unit": "canvas passes/s",
                                "cores": smp.cores(), "kind": "oracle", "sample": smp.describe()}
    print(json.dumps(line))
    if ws_ > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
