"""B300-native canvas pass of a uniform-state block text-diffusion sampler.

A thin ctypes binding over libdgcanvas.so (C ABI in include/dgcanvas.h). Every step of the
path -- the vocabulary-head contraction with its fused softmax statistics, the confidence top-K
keep, the counter-hash re-randomisation, the stop test and the graph-driven loop -- runs in the
library's CUDA kernels; this module only marshals torch tensors, streams and structs. There is
no CPU fallback: if the library or a CUDA device is missing, calls raise.

Names mirror the C entry points: dg_workspace_bytes, dg_canvas_stats, dg_canvas_step,
dg_canvas_loop (plus dg_synth_denoise as the built-in denoiser hook).
"""
from __future__ import annotations

import ctypes as C
import itertools
from pathlib import Path

import torch

__all__ = ["DG_F32", "DG_BF16", "DG_E4M3", "HeadDesc", "CanvasState", "StopRule", "LoopParams",
           "SynthParams", "DgError", "lib", "dg_workspace_bytes", "dg_canvas_stats",
           "dg_canvas_step", "dg_canvas_loop", "dg_status_string", "dtype_code", "new_state",
           "REASON_ENTROPY", "REASON_STABLE", "REASON_CAP", "ST_BAD_TOKEN", "ST_NONFINITE",
           "ST_TIMEOUT", "STOP_OR", "STOP_AND", "KEEP_CONFIDENCE", "KEEP_ENTROPY",
           "REDRAW_UNIFORM", "REDRAW_MASK", "pass_rule", "dg_block_generate", "timeline_us",
           "DG_NVFP4", "nvfp4_scale_bytes", "dg_nvfp4_pack_scales", "dg_quantize_nvfp4",
           "dg_profile_next_head", "dg_profile_next_head_clock", "sm_clock_stats",
           "dg_selftest_wait_timeout", "dg_quantize_e4m3"]

DG_F32, DG_BF16, DG_E4M3, DG_NVFP4 = 0, 1, 2, 3
DG_TL_DENOISE, DG_TL_HEAD, DG_TL_MERGE, DG_TL_KERNELS = 0, 1, 2, 3
REASON_ENTROPY, REASON_STABLE, REASON_CAP = 1, 2, 4
ST_BAD_TOKEN, ST_NONFINITE, ST_TIMEOUT = 1, 2, 4
STOP_OR, STOP_AND = 0, 1
KEEP_CONFIDENCE, KEEP_ENTROPY = 0, 1
REDRAW_UNIFORM, REDRAW_MASK = 0, 1

_LIB_PATH = Path(__file__).resolve().parent / "libdgcanvas.so"
_lib = None


class DgError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {dg_status_string(code)} ({code})")


class HeadDesc(C.Structure):
    _fields_ = [("B", C.c_int32), ("S", C.c_int32), ("d", C.c_int32), ("V", C.c_int32),
                ("h_dtype", C.c_int32), ("w_dtype", C.c_int32), ("h", C.c_void_p),
                ("h_scale", C.c_void_p), ("w", C.c_void_p), ("w_scale", C.c_void_p),
                ("inv_temp", C.c_float), ("h_block_scale", C.c_void_p),
                ("w_block_scale", C.c_void_p)]


class CanvasState(C.Structure):
    _fields_ = [("passes", C.c_int32), ("reason", C.c_int32), ("stable", C.c_int32),
                ("done", C.c_int32), ("mean_entropy", C.c_float), ("last_pass", C.c_int32),
                ("reserved", C.c_int32 * 2)]


class StopRule(C.Structure):
    _fields_ = [("max_passes", C.c_int32), ("entropy_threshold", C.c_float),
                ("stable_passes", C.c_int32), ("stop_mode", C.c_int32), ("keep_rule", C.c_int32),
                ("redraw_mode", C.c_int32), ("mask_id", C.c_int32)]


class LoopParams(C.Structure):
    _fields_ = [("rule", StopRule), ("keep_k0", C.c_int32), ("keep_sched", C.c_void_p),
                ("seed", C.c_uint64), ("start_pass", C.c_uint32), ("init_random", C.c_uint32),
                ("trace_mean_entropy", C.c_void_p), ("trace_canvas", C.c_void_p),
                ("trace_h", C.c_void_p), ("trace_argmax", C.c_void_p), ("trace_conf", C.c_void_p),
                ("trace_entropy", C.c_void_p), ("trace_timeline", C.c_void_p),
                ("temp_start", C.c_float), ("temp_end", C.c_float), ("row_offset", C.c_uint64),
                ("trace_sm_clock", C.c_void_p)]


class SynthParams(C.Structure):
    _fields_ = [("desc", C.POINTER(HeadDesc)), ("y", C.c_void_p), ("n_content", C.c_int32),
                ("s_content", C.c_float), ("s_pad", C.c_float), ("status", C.c_void_p)]


_HOOK_TOKENS = itertools.count(1)

DENOISE_FN = C.CFUNCTYPE(C.c_int, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p)


def lib():
    """Load libdgcanvas.so (built in-tree by uniform_state_denoising_vocab_b300.build)."""
    global _lib
    if _lib is None:
        if not _LIB_PATH.exists():
            raise ImportError(f"libdgcanvas.so not built at {_LIB_PATH}; run "
                              "`python -m uniform_state_denoising_vocab_b300.build`")
        L = C.CDLL(str(_LIB_PATH))
        vp, sz = C.c_void_p, C.c_size_t
        L.dg_workspace_bytes.argtypes = [C.POINTER(HeadDesc), C.POINTER(sz)]
        L.dg_canvas_stats.argtypes = [C.POINTER(HeadDesc), vp, vp, vp, vp, vp, sz, vp, vp]
        L.dg_canvas_step.argtypes = [C.POINTER(HeadDesc), vp, vp, C.c_int32, C.c_uint64,
                                     C.c_uint32, vp, vp, vp, vp, vp, vp, C.POINTER(StopRule), vp,
                                     sz, vp, vp]
        L.dg_canvas_loop.argtypes = [C.POINTER(HeadDesc), vp, vp, C.POINTER(LoopParams), vp, vp,
                                     vp, vp, vp, vp, vp, sz, vp, vp]
        L.dg_status_string.argtypes = [C.c_int]
        L.dg_status_string.restype = C.c_char_p
        L.dg_version.restype = C.c_int
        L.dg_nvfp4_scale_bytes.argtypes = [C.c_int32, C.c_int32, C.POINTER(sz)]
        L.dg_nvfp4_pack_scales.argtypes = [vp, C.c_int32, C.c_int32, vp, vp]
        L.dg_quantize_nvfp4.argtypes = [vp, C.c_int32, C.c_int32, vp, vp, vp, vp, vp]
        for f in ("dg_nvfp4_scale_bytes", "dg_nvfp4_pack_scales", "dg_quantize_nvfp4"):
            getattr(L, f).restype = C.c_int
        L.dg_block_generate.argtypes = [C.POINTER(HeadDesc), C.c_int32, vp, vp, vp, vp, vp,
                                        C.POINTER(LoopParams), C.c_int32, C.c_float, C.c_float,
                                        vp, vp, vp, sz, vp, vp]
        L.dg_block_generate.restype = C.c_int
        L.dg_workspace_bytes_host.argtypes = [C.POINTER(HeadDesc), C.POINTER(sz)]
        L.dg_workspace_bytes_host.restype = C.c_int
        L.dg_canvas_step_host.argtypes = [C.POINTER(HeadDesc), vp, vp, vp, C.c_int32, C.c_uint64,
                                          C.c_uint32, vp, C.POINTER(StopRule), vp, sz, vp, vp]
        L.dg_canvas_step_host.restype = C.c_int
        L.dg_profile_next_head.argtypes = [C.c_void_p, C.c_void_p]
        L.dg_profile_next_head.restype = C.c_int
        L.dg_profile_next_head_clock.argtypes = [C.c_void_p]
        L.dg_profile_next_head_clock.restype = C.c_int
        L.dg_quantize_e4m3.argtypes = [vp, C.c_int32, C.c_int32, vp, vp, vp, vp]
        L.dg_quantize_e4m3.restype = C.c_int
        L.dg_selftest_wait_timeout.argtypes = [C.c_void_p, C.c_void_p]
        L.dg_selftest_wait_timeout.restype = C.c_int
        for f in ("dg_workspace_bytes", "dg_canvas_stats", "dg_canvas_step", "dg_canvas_loop"):
            getattr(L, f).restype = C.c_int
        _lib = L
    return _lib


def dg_profile_next_head(start: torch.cuda.Event, stop: torch.cuda.Event) -> None:
    """Bracket the next head kernel launched by this thread with two recorded CUDA events."""
    for ev in (start, stop):
        if not ev.cuda_event:   # torch creates the cudaEvent_t lazily, at its first record
            ev.record()
    _check(lib().dg_profile_next_head(C.c_void_p(start.cuda_event), C.c_void_p(stop.cuda_event)),
           "dg_profile_next_head")


def dg_profile_next_head_clock(sample: torch.Tensor) -> None:
    """Have the next head kernel launched by this thread write its SM clock sample into
    `sample` (device int64 [4]: clock64 and global-timer ns at begin, then at end)."""
    if sample.numel() < 4 or sample.element_size() != 8:
        raise ValueError("the clock sample needs 4 x 8 bytes")
    _check(lib().dg_profile_next_head_clock(_ptr(sample)), "dg_profile_next_head_clock")


def sm_clock_stats(samples) -> dict:
    """Effective SM clock (MHz) and head duration in SM cycles from clock samples [n, 4]
    (rows with no sample are skipped)."""
    t = samples.detach().cpu().view(-1, 4).numpy().view("uint64").astype("float64")
    ok = (t[:, 3] > t[:, 1]) & (t[:, 2] > t[:, 0])
    t = t[ok]
    if not len(t):
        return {"sm_mhz_effective": None, "head_kcycles": None, "samples": 0}
    mhz = (t[:, 2] - t[:, 0]) / (t[:, 3] - t[:, 1]) * 1e3
    import statistics
    return {"sm_mhz_effective": round(statistics.median(mhz.tolist()), 1),
            "head_kcycles": round(statistics.median(((t[:, 2] - t[:, 0]) / 1e3).tolist()), 2),
            "samples": int(len(t))}


def dg_selftest_wait_timeout(status=None, stream=None) -> torch.Tensor:
    """Launch the library's self-test of its bounded waits: one kernel whose only wait can never
    complete gives up after the wall-time bound (about 2 s) and sets ST_TIMEOUT in the returned
    status word (enqueued on `stream`; synchronise before reading it)."""
    st = torch.zeros(1, dtype=torch.int32, device="cuda") if status is None else status
    _check(lib().dg_selftest_wait_timeout(_ptr(st), _stream(stream)), "dg_selftest_wait_timeout")
    return st


def dg_status_string(code: int) -> str:
    return lib().dg_status_string(int(code)).decode()


def _check(rc: int, where: str) -> None:
    if rc != 0:
        raise DgError(rc, where)


def dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return DG_F32
    if t.dtype == torch.bfloat16:
        return DG_BF16
    if t.dtype in (torch.float8_e4m3fn, torch.uint8):
        return DG_E4M3
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to libdgcanvas must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors passed to libdgcanvas must be contiguous")
    return C.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def make_desc(h, w, *, B: int, S: int, h_scale=None, w_scale=None, inv_temp: float = 1.0,
              h_dtype: int | None = None, d: int | None = None, w_dtype: int | None = None,
              h_block_scale=None, w_block_scale=None) -> HeadDesc:
    """Head descriptor over torch tensors: h [B*S, d] (or None for a loop's buffer later),
    w [V, d], optional fp32 scales for E4M3 / NVFP4 operands. NVFP4 operands are uint8 code
    tensors [rows, d/2] with w_dtype / h_dtype = DG_NVFP4 and packed block scales."""
    V, dd = int(w.shape[0]), int(w.shape[1])
    wd = dtype_code(w) if w_dtype is None else w_dtype
    if wd == DG_NVFP4:
        dd *= 2
    hd = (h_dtype if h_dtype is not None else dtype_code(h)) if h is not None else \
        (DG_BF16 if h_dtype is None else h_dtype)
    d_ = dd if d is None else d
    desc = HeadDesc(B=B, S=S, d=d_, V=V, h_dtype=hd, w_dtype=wd,
                    h=None if h is None else _ptr(h).value, h_scale=None if h_scale is None else
                    _ptr(h_scale).value, w=_ptr(w).value,
                    w_scale=None if w_scale is None else _ptr(w_scale).value,
                    inv_temp=float(inv_temp))
    desc.h_block_scale = None if h_block_scale is None else _ptr(h_block_scale).value
    desc.w_block_scale = None if w_block_scale is None else _ptr(w_block_scale).value
    return desc


def dg_workspace_bytes(desc: HeadDesc) -> int:
    n = C.c_size_t(0)
    _check(lib().dg_workspace_bytes(C.byref(desc), C.byref(n)), "dg_workspace_bytes")
    return int(n.value)


def _workspace(desc: HeadDesc, device, workspace=None):
    need = dg_workspace_bytes(desc)
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < need:
            raise ValueError(f"workspace too small: need {need} bytes")
        return workspace
    return torch.empty(max(need, 256), dtype=torch.uint8, device=device)


def new_state(B: int, device) -> torch.Tensor:
    """Device array of B dg_canvas_state records (8 int32 each), zero-initialised."""
    return torch.zeros(B, 8, dtype=torch.int32, device=device)


def nvfp4_scale_bytes(rows: int, d: int) -> int:
    n = C.c_size_t(0)
    _check(lib().dg_nvfp4_scale_bytes(int(rows), int(d), C.byref(n)), "dg_nvfp4_scale_bytes")
    return int(n.value)


def dg_nvfp4_pack_scales(block_scales, rows: int, d: int, stream=None) -> torch.Tensor:
    """Plain E4M3 block scales [rows, d/16] (uint8, device) -> the packed layout NVFP4 heads read."""
    out = torch.empty(nvfp4_scale_bytes(rows, d), dtype=torch.uint8, device=block_scales.device)
    _check(lib().dg_nvfp4_pack_scales(_ptr(block_scales), int(rows), int(d), _ptr(out),
                                      _stream(stream)), "dg_nvfp4_pack_scales")
    return out


def dg_quantize_e4m3(h, status=None, stream=None) -> dict:
    """Per-row E4M3 quantisation of bf16 h [rows, d] on the device: codes (uint8 [rows, d]) and
    row scales (fp32 [rows]), the rule a (BF16, E4M3) pass applies to its hidden states."""
    rows, d = int(h.shape[0]), int(h.shape[1])
    dev = h.device
    out = {"codes": torch.empty(rows, d, dtype=torch.uint8, device=dev),
           "scale": torch.empty(rows, dtype=torch.float32, device=dev),
           "status": torch.zeros(1, dtype=torch.int32, device=dev) if status is None else status}
    _check(lib().dg_quantize_e4m3(_ptr(h), rows, d, _ptr(out["codes"]), _ptr(out["scale"]),
                                  _ptr(out["status"]), _stream(stream)), "dg_quantize_e4m3")
    return out


def dg_quantize_nvfp4(h, status=None, stream=None) -> dict:
    """NVFP4 quantisation of bf16 rows h [rows, d] on the device: codes [rows, d/2], packed block
    scales and fp32 row scales [rows]."""
    rows, d = int(h.shape[0]), int(h.shape[1])
    dev = h.device
    out = {"codes": torch.empty(rows, d // 2, dtype=torch.uint8, device=dev),
           "block_scale": torch.empty(nvfp4_scale_bytes(rows, d), dtype=torch.uint8, device=dev),
           "scale": torch.empty(rows, dtype=torch.float32, device=dev),
           "status": torch.zeros(1, dtype=torch.int32, device=dev) if status is None else status}
    _check(lib().dg_quantize_nvfp4(_ptr(h), rows, d, _ptr(out["codes"]), _ptr(out["block_scale"]),
                                   _ptr(out["scale"]), _ptr(out["status"]), _stream(stream)),
           "dg_quantize_nvfp4")
    return out


def dg_canvas_stats(h, w, *, B: int, S: int, h_scale=None, w_scale=None, inv_temp: float = 1.0,
                    workspace=None, status=None, stream=None, **desc_kw) -> dict:
    """Per-slot argmax, confidence (max prob), entropy (nats) and per-canvas mean entropy."""
    dev = w.device
    R = B * S
    desc = make_desc(h, w, B=B, S=S, h_scale=h_scale, w_scale=w_scale, inv_temp=inv_temp, **desc_kw)
    ws = _workspace(desc, dev, workspace)
    out = {"argmax": torch.empty(R, dtype=torch.int32, device=dev),
           "conf": torch.empty(R, dtype=torch.float32, device=dev),
           "entropy": torch.empty(R, dtype=torch.float32, device=dev),
           "mean_entropy": torch.empty(B, dtype=torch.float32, device=dev)}
    st = torch.zeros(1, dtype=torch.int32, device=dev) if status is None else status
    rc = lib().dg_canvas_stats(C.byref(desc), _ptr(out["argmax"]), _ptr(out["conf"]),
                               _ptr(out["entropy"]), _ptr(out["mean_entropy"]), _ptr(ws),
                               ws.numel(), _ptr(st), _stream(stream))
    _check(rc, "dg_canvas_stats")
    out["status"] = st
    return out


def _host_ptr(t):
    if t is None:
        return None
    if t.device.type != "cpu":
        raise ValueError("host buffers of dg_canvas_step_host must be CPU tensors")
    if not t.is_contiguous():
        raise ValueError("tensors passed to libdgcanvas must be contiguous")
    return C.c_void_p(t.data_ptr())


def host_desc(h, w, *, B: int, S: int, h_scale=None, h_block_scale=None, w_scale=None,
              inv_temp: float = 1.0, **desc_kw) -> HeadDesc:
    """Head descriptor whose h (and h_scale / h_block_scale) are host tensors, w on the device."""
    hd = dtype_code(h) if "h_dtype" not in desc_kw else desc_kw.pop("h_dtype")
    d_ = desc_kw.pop("d", None)
    if d_ is None:
        d_ = int(h.shape[1]) * (2 if hd == DG_NVFP4 else 1)
    desc = make_desc(None, w, B=B, S=S, w_scale=w_scale, inv_temp=inv_temp, h_dtype=hd, d=d_,
                     **desc_kw)
    desc.h = _host_ptr(h).value
    desc.h_scale = None if h_scale is None else _host_ptr(h_scale).value
    desc.h_block_scale = None if h_block_scale is None else _host_ptr(h_block_scale).value
    return desc


def dg_workspace_bytes_host(desc: HeadDesc) -> int:
    n = C.c_size_t(0)
    _check(lib().dg_workspace_bytes_host(C.byref(desc), C.byref(n)), "dg_workspace_bytes_host")
    return int(n.value)


def dg_canvas_step_host(h, w, canvas_in, keep_k: int, seed: int, pass_: int, *, B: int, S: int,
                        canvas_out=None, mean_entropy=None, h_scale=None, h_block_scale=None,
                        w_scale=None, inv_temp: float = 1.0, state=None,
                        rule: StopRule | None = None, workspace=None, status=None, stream=None,
                        desc: HeadDesc | None = None, **desc_kw) -> dict:
    """One canvas pass on host buffers: h [B*S, d] (and its scales) and canvas_in [B*S] are CPU
    tensors (page-locked for asynchronous copies); the new canvas and the per-canvas mean entropy
    are written to CPU tensors, valid once `stream` has synchronised. w stays on the device.
    Pass a prebuilt `desc` (host_desc) and `workspace` to avoid per-call set-up."""
    dev = w.device
    if desc is None:
        desc = host_desc(h, w, B=B, S=S, h_scale=h_scale, h_block_scale=h_block_scale,
                         w_scale=w_scale, inv_temp=inv_temp, **desc_kw)
    if workspace is None:
        workspace = torch.empty(dg_workspace_bytes_host(desc), dtype=torch.uint8, device=dev)
    R = B * S
    if canvas_out is None:
        canvas_out = torch.empty(R, dtype=torch.int32).pin_memory()
    if mean_entropy is None:
        mean_entropy = torch.empty(B, dtype=torch.float32).pin_memory()
    st = torch.zeros(1, dtype=torch.int32, device=dev) if status is None else status
    rc = lib().dg_canvas_step_host(C.byref(desc), _host_ptr(canvas_in), _host_ptr(canvas_out),
                                   _host_ptr(mean_entropy), int(keep_k), C.c_uint64(seed),
                                   C.c_uint32(pass_ & 0xFFFFFFFF), _ptr(state),
                                   None if rule is None else C.byref(rule), _ptr(workspace),
                                   workspace.numel(), _ptr(st), _stream(stream))
    _check(rc, "dg_canvas_step_host")
    return {"canvas": canvas_out, "mean_entropy": mean_entropy, "status": st}


def pass_rule(keep_rule: int = KEEP_CONFIDENCE, mask_id: int | None = None,
              base: StopRule | None = None) -> StopRule:
    """A rule carrying a pass's keep / re-draw variant (and, from `base`, its stop test)."""
    r = StopRule(max_passes=1 << 30, entropy_threshold=0.0, stable_passes=1 << 30,
                 stop_mode=STOP_OR) if base is None else StopRule.from_buffer_copy(base)
    r.keep_rule = keep_rule
    r.redraw_mode = REDRAW_UNIFORM if mask_id is None else REDRAW_MASK
    r.mask_id = 0 if mask_id is None else int(mask_id)
    return r


def dg_canvas_step(h, w, canvas_in, keep_k: int, seed: int, pass_: int, *, B: int, S: int,
                   canvas_out=None, h_scale=None, w_scale=None, inv_temp: float = 1.0,
                   state=None, rule: StopRule | None = None, keep_rule: int = KEEP_CONFIDENCE,
                   mask_id: int | None = None, outputs: bool = True, workspace=None, status=None,
                   stream=None, **desc_kw) -> dict:
    """One canvas pass: statistics, keep the top-K by confidence (or the K lowest-entropy slots
    with keep_rule=KEEP_ENTROPY), re-randomise the rest (or set them to mask_id)."""
    if rule is None and (keep_rule != KEEP_CONFIDENCE or mask_id is not None):
        rule = pass_rule(keep_rule, mask_id)
    dev = w.device
    R = B * S
    desc = make_desc(h, w, B=B, S=S, h_scale=h_scale, w_scale=w_scale, inv_temp=inv_temp, **desc_kw)
    ws = _workspace(desc, dev, workspace)
    out = {"canvas": canvas_out if canvas_out is not None else torch.empty(R, dtype=torch.int32, device=dev)}
    if outputs:
        out.update({"argmax": torch.empty(R, dtype=torch.int32, device=dev),
                    "conf": torch.empty(R, dtype=torch.float32, device=dev),
                    "entropy": torch.empty(R, dtype=torch.float32, device=dev),
                    "kept": torch.empty(R, dtype=torch.uint8, device=dev),
                    "mean_entropy": torch.empty(B, dtype=torch.float32, device=dev)})
    g = out.get
    st = torch.zeros(1, dtype=torch.int32, device=dev) if status is None else status
    rc = lib().dg_canvas_step(C.byref(desc), _ptr(canvas_in), _ptr(out["canvas"]), int(keep_k),
                              C.c_uint64(seed), C.c_uint32(pass_ & 0xFFFFFFFF), _ptr(g("argmax")),
                              _ptr(g("conf")), _ptr(g("entropy")), _ptr(g("kept")),
                              _ptr(g("mean_entropy")), _ptr(state),
                              None if rule is None else C.byref(rule), _ptr(ws), ws.numel(),
                              _ptr(st), _stream(stream))
    _check(rc, "dg_canvas_step")
    out["status"] = st
    return out


def prepare_loop(w, canvas, *, B: int, S: int, theta: float, y=None, denoise=None,
                   h_buffer=None, w_scale=None, keep_k0: int = 32, keep_sched=None,
                   seed: int = 0, max_passes: int = 48, stable_passes: int = 2,
                   stop_mode: int = STOP_OR, start_pass: int = 0, init_random: bool = True,
                   state=None, n_content: int = 50, s_content: float = 8.0, s_pad: float = 16.0,
                   trace: bool = False, timeline: bool = False, sm_clock: bool = False,
                   workspace=None, status=None,
                   outputs: dict | None = None, keep_rule: int = KEEP_CONFIDENCE,
                   mask_id: int | None = None, temp_start: float = 0.0, temp_end: float = 0.0,
                   row_offset: int = 0) -> "PreparedLoop":
    """Marshal the arguments of a dg_canvas_loop call once; PreparedLoop.run(stream) issues it
    (again and again: the library reuses its captured graph while the arguments are unchanged).

    With y given (and denoise None) the built-in synthetic denoiser is used. `denoise`, if
    given, is a Python callable (canvas_ptr, pass_ptr, h_ptr, stream_handle) -> int that must
    enqueue capturable work on the stream it receives; it is called while the library captures
    the loop (once per prepared call, on its first run), and later runs replay that work. `outputs` may hold preallocated
    argmax/conf/entropy tensors [B*S]; with the same tensors (and the same other arguments) a
    repeated call reuses the captured graph. With timeline=True the result holds
    "trace_timeline" [max_passes, 3, 2] (uint64 stored as int64): per pass, the device global
    timer (ns) at the begin/end of the denoiser (built-in only), the head and the merge kernel.
    With sm_clock=True it holds "trace_sm_clock" [max_passes, 4]: each pass's head clock sample
    (sm_clock_stats turns it into the effective SM clock and the head's cycle count).
    """
    dev = w.device
    R = B * S
    d = int(w.shape[1])
    if h_buffer is None:
        h_buffer = torch.empty(R, d, dtype=torch.bfloat16, device=dev)
    desc = make_desc(h_buffer, w, B=B, S=S, w_scale=w_scale)
    ws = _workspace(desc, dev, workspace)
    if state is None:
        state = new_state(B, dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev) if status is None else status
    outputs = outputs or {}
    out = {"canvas": canvas, "state": state, "status": st, "h": h_buffer,
           "argmax": outputs.get("argmax", None), "conf": outputs.get("conf", None),
           "entropy": outputs.get("entropy", None)}
    if out["argmax"] is None:
        out["argmax"] = torch.empty(R, dtype=torch.int32, device=dev)
    for k in ("conf", "entropy"):
        if out[k] is None:
            out[k] = torch.empty(R, dtype=torch.float32, device=dev)
    params = LoopParams(rule=pass_rule(keep_rule, mask_id,
                                       StopRule(max_passes=max_passes, entropy_threshold=theta,
                                                stable_passes=stable_passes, stop_mode=stop_mode)),
                        temp_start=temp_start, temp_end=temp_end, row_offset=row_offset,
                        keep_k0=keep_k0, keep_sched=None if keep_sched is None else _ptr(keep_sched).value,
                        seed=seed, start_pass=start_pass, init_random=1 if init_random else 0)
    if trace:
        out["trace_mean_entropy"] = torch.full((max_passes, B), float("nan"), device=dev)
        out["trace_canvas"] = torch.full((max_passes, R), -1, dtype=torch.int32, device=dev)
        out["trace_h"] = torch.zeros(max_passes, R, d, dtype=h_buffer.dtype, device=dev)
        params.trace_mean_entropy = _ptr(out["trace_mean_entropy"]).value
        params.trace_canvas = _ptr(out["trace_canvas"]).value
        params.trace_h = _ptr(out["trace_h"]).value
        out["trace_argmax"] = torch.full((max_passes, R), -1, dtype=torch.int32, device=dev)
        out["trace_conf"] = torch.full((max_passes, R), float("nan"), device=dev)
        out["trace_entropy"] = torch.full((max_passes, R), float("nan"), device=dev)
        params.trace_argmax = _ptr(out["trace_argmax"]).value
        params.trace_conf = _ptr(out["trace_conf"]).value
        params.trace_entropy = _ptr(out["trace_entropy"]).value
    if timeline:
        out["trace_timeline"] = torch.empty(max_passes, DG_TL_KERNELS, 2, dtype=torch.int64, device=dev)
        params.trace_timeline = _ptr(out["trace_timeline"]).value
    if sm_clock:
        out["trace_sm_clock"] = torch.zeros(max_passes, 4, dtype=torch.int64, device=dev)
        params.trace_sm_clock = _ptr(out["trace_sm_clock"]).value
    L = lib()
    keep = []
    if denoise is None:
        if y is None:
            raise ValueError("give y (synthetic denoiser) or a denoise callable")
        sp = SynthParams(desc=C.pointer(desc), y=_ptr(y).value, n_content=n_content,
                         s_content=s_content, s_pad=s_pad, status=_ptr(st).value)
        fn = C.cast(L.dg_synth_denoise, C.c_void_p)
        user = C.cast(C.pointer(sp), C.c_void_p)
        keep += [sp]
    else:
        cb = DENOISE_FN(lambda u, c, p, h, s: int(denoise(c, p, h, s) or 0))
        fn = C.cast(cb, C.c_void_p)
        # The library caches the captured loop per (hook, user): a fresh token per prepared call
        # keeps a later callback whose trampoline reuses a freed address from replaying this one.
        user = C.c_void_p(next(_HOOK_TOKENS))
        keep += [cb]
    call = (C.byref(desc), _ptr(canvas), _ptr(h_buffer), C.byref(params), fn, user, _ptr(state),
            _ptr(out["argmax"]), _ptr(out["conf"]), _ptr(out["entropy"]), _ptr(ws), ws.numel(),
            _ptr(st))
    out["_keepalive"] = keep + [ws, desc, params]
    return PreparedLoop(call, out)


class PreparedLoop:
    """One dg_canvas_loop call with its arguments marshalled (see prepare_loop)."""

    def __init__(self, call, out):
        self._call = call
        self.out = out

    def run(self, stream=None) -> dict:
        _check(lib().dg_canvas_loop(*self._call, _stream(stream)), "dg_canvas_loop")
        return self.out


def dg_canvas_loop(w, canvas, *, stream=None, **kw) -> dict:
    """The whole denoising loop on the device (one graph launch, no host synchronisation): the
    keyword arguments of prepare_loop, issued once on `stream`."""
    return prepare_loop(w, canvas, **kw).run(stream)


def dg_block_generate(w, y_blocks, *, n_blocks: int, B: int, S: int, theta: float,
                      w_scale=None, keep_k0: int = 32, seed: int = 0, max_passes: int = 48,
                      stable_passes: int = 2, stop_mode: int = STOP_OR, n_content: int = 50,
                      s_content: float = 8.0, s_pad: float = 16.0, keep_rule: int = KEEP_CONFIDENCE,
                      mask_id: int | None = None, temp_start: float = 0.0, temp_end: float = 0.0,
                      row_offset: int = 0, workspace=None, status=None, stream=None) -> dict:
    """Block-autoregressive generation with the built-in synthetic denoiser: n_blocks loops, one
    per block of B*S slots with targets y_blocks[i], each committing its final canvas."""
    dev = w.device
    R = B * S
    d = int(w.shape[1])
    h_buffer = torch.empty(R, d, dtype=torch.bfloat16, device=dev)
    desc = make_desc(h_buffer, w, B=B, S=S, w_scale=w_scale)
    ws = _workspace(desc, dev, workspace)
    st = torch.zeros(1, dtype=torch.int32, device=dev) if status is None else status
    out = {"tokens": torch.empty(n_blocks * R, dtype=torch.int32, device=dev),
           "states": torch.zeros(n_blocks * B, 8, dtype=torch.int32, device=dev), "status": st}
    y_work = torch.empty(R, dtype=torch.int32, device=dev)
    canvas = torch.empty(R, dtype=torch.int32, device=dev)
    state = new_state(B, dev)
    params = LoopParams(rule=pass_rule(keep_rule, mask_id,
                                       StopRule(max_passes=max_passes, entropy_threshold=theta,
                                                stable_passes=stable_passes, stop_mode=stop_mode)),
                        keep_k0=keep_k0, seed=seed, temp_start=temp_start, temp_end=temp_end,
                        row_offset=row_offset)
    rc = lib().dg_block_generate(C.byref(desc), int(n_blocks), _ptr(y_blocks), _ptr(y_work),
                                 _ptr(canvas), _ptr(state), _ptr(h_buffer), C.byref(params),
                                 int(n_content), float(s_content), float(s_pad),
                                 _ptr(out["tokens"]), _ptr(out["states"]), _ptr(ws), ws.numel(),
                                 _ptr(st), _stream(stream))
    _check(rc, "dg_block_generate")
    out["_keepalive"] = [ws, desc, params, y_work, canvas, state, h_buffer]
    return out


def timeline_us(tl: torch.Tensor, passes: int) -> list:
    """Per-pass kernel intervals in microseconds relative to the first recorded stamp, from a
    loop's "trace_timeline": [{"denoise": (b, e) | None, "head": (b, e), "merge": (b, e)}, ...]."""
    t = tl.detach().cpu().view(-1, DG_TL_KERNELS, 2).numpy().view("uint64")
    valid = t[:passes][t[:passes, :, 1] > 0]
    t0 = int(valid[:, 0].min()) if valid.size else 0
    names = ("denoise", "head", "merge")
    out = []
    for p in range(passes):
        row = {}
        for k, n in enumerate(names):
            b, e = int(t[p, k, 0]), int(t[p, k, 1])
            row[n] = None if e == 0 else ((b - t0) / 1e3, (e - t0) / 1e3)
        out.append(row)
    return out


def state_fields(state: torch.Tensor) -> dict:
    """Decode a [B, 8] int32 state tensor (host copy) into named fields."""
    s = state.detach().cpu()
    return {"passes": s[:, 0].clone(), "reason": s[:, 1].clone(), "stable": s[:, 2].clone(),
            "done": s[:, 3].clone(), "mean_entropy": s[:, 4].view(torch.float32).clone(),
            "last_pass": s[:, 5].clone()}
