"""ctypes wrapper around dg_oracle.c plus the loop control, written plainly in Python.

TEST INFRASTRUCTURE ONLY: the checker for the CUDA library, never a fallback for it.

The per-pass arithmetic (logits in double, two-pass softmax, sort-based top-K, SplitMix64 draws,
E4M3/bf16 rounding, the synthetic denoiser) is in dg_oracle.c; this file builds that library with
gcc, marshals numpy arrays, and runs the denoising loop:

  start from a canvas of random vocabulary tokens; on every pass p (t = p + 1) denoise the canvas
  into hidden states, predict every slot, keep the K_t most confident slots at their argmax and
  re-draw the others uniformly ("When to use a diffusion LLM" (devengoratela.com), "How block
  diffusion works"); stop when the mean canvas entropy falls below a threshold, when the canvas
  has been unchanged for two consecutive passes, or after 48 passes ("DiffusionGemma 26B: How
  Google's Text Diffusion Model Generates Tokens in Parallel" (dev.to), "How Diffusion Changes the
  Equation").
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from pathlib import Path

import numpy as np

OR_F32, OR_BF16, OR_E4M3, OR_NVFP4 = 0, 1, 2, 3
_DT = {"f32": OR_F32, "bf16": OR_BF16, "e4m3": OR_E4M3, "nvfp4": OR_NVFP4, OR_F32: OR_F32,
       OR_BF16: OR_BF16, OR_E4M3: OR_E4M3, OR_NVFP4: OR_NVFP4}

INIT_PASS = 0xFFFFFFFF          # hash pass index of the initial random canvas
REASON_ENTROPY, REASON_STABLE, REASON_CAP = 1, 2, 4

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "dg_oracle.c"
_LIB_PATH = _HERE / "_build" / "liboracle.so"
_lib = None


def build(force: bool = False) -> Path:
    """Compile dg_oracle.c with gcc (-O2, OpenMP, no floating-point contraction)."""
    _LIB_PATH.parent.mkdir(parents=True, exist_ok=True)
    if force or not _LIB_PATH.exists() or _LIB_PATH.stat().st_mtime < _SRC.stat().st_mtime:
        tmp = _LIB_PATH.with_suffix(f".{os.getpid()}.tmp")
        subprocess.run(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-std=c11", "-shared",
                        "-fPIC", "-o", str(tmp), str(_SRC), "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    if _lib is None:
        lib = C.CDLL(str(build()))
        i64, u64, u32, vp, dbl = C.c_int64, C.c_uint64, C.c_uint32, C.c_void_p, C.c_double
        lib.or_head_stats.argtypes = [i64, i64, i64, C.c_int, vp, vp, vp, vp, dbl, vp, i64,
                                      vp, vp, vp, vp, vp, vp]
        lib.or_head_stats.restype = C.c_int
        lib.or_select.argtypes = [i64, i64, i64, vp, vp, vp, i64, u64, u32, C.c_int, i64, u64,
                                  vp, vp, vp, vp]
        lib.or_select.restype = C.c_int
        lib.or_sm64.argtypes = [u64]
        lib.or_sm64.restype = u64
        lib.or_key.argtypes = [u64, u32, u64]
        lib.or_key.restype = u64
        lib.or_draw.argtypes = [u64, u32, u64, i64]
        lib.or_draw.restype = C.c_int32
        lib.or_keys.argtypes = [u64, u32, vp, i64, vp]
        lib.or_sm64_many.argtypes = [vp, i64, vp]
        lib.or_bf16_round_many.argtypes = [vp, i64, vp]
        lib.or_e4m3_round_many.argtypes = [vp, i64, vp]
        lib.or_e4m3_value_many.argtypes = [vp, i64, vp]
        lib.or_quant_rows_e4m3.argtypes = [vp, i64, i64, vp, vp]
        lib.or_quant_rows_nvfp4.argtypes = [vp, i64, i64, vp, vp, vp]
        lib.or_e2m1_round_many.argtypes = [vp, i64, vp]
        lib.or_e2m1_value_many.argtypes = [vp, i64, vp]
        lib.or_synth_denoise.argtypes = [i64, i64, i64, i64, C.c_int, vp, vp, vp, vp, u32, i64,
                                         dbl, dbl, vp]
        lib.or_synth_denoise.restype = C.c_int
        lib.or_num_threads.restype = C.c_int
        _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


def _operand(dtype: int, a):
    return _c(a, {OR_F32: np.float32, OR_BF16: np.uint16, OR_E4M3: np.uint8,
                  OR_NVFP4: np.uint8}[dtype])


def _elems(dtype: int, a) -> int:
    """Number of operand elements in a stored array (NVFP4 packs two per byte)."""
    return a.size * 2 if dtype == OR_NVFP4 else a.size


def num_threads() -> int:
    return int(_L().or_num_threads())


# ---------------------------------------------------------------------------------------------
# number formats and hash
# ---------------------------------------------------------------------------------------------
def sm64(x) -> np.ndarray:
    x = _c(np.atleast_1d(x), np.uint64)
    out = np.empty_like(x)
    _L().or_sm64_many(_p(x), x.size, _p(out))
    return out


def keys(seed: int, pass_: int, rows) -> np.ndarray:
    rows = _c(np.atleast_1d(rows), np.uint64)
    out = np.empty_like(rows)
    _L().or_keys(C.c_uint64(seed), C.c_uint32(pass_ & 0xFFFFFFFF), _p(rows), rows.size, _p(out))
    return out


def draw(seed: int, pass_: int, rows, V: int) -> np.ndarray:
    """Uniform vocabulary draws key(seed, pass, row) mod V."""
    return (keys(seed, pass_, rows) % np.uint64(V)).astype(np.int32)


def bf16_round(x) -> np.ndarray:
    x = _c(x, np.float64)
    out = np.empty(x.shape, np.uint16)
    _L().or_bf16_round_many(_p(x), x.size, _p(out))
    return out


def e4m3_round(x) -> np.ndarray:
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    _L().or_e4m3_round_many(_p(x), x.size, _p(out))
    return out


def e4m3_value(q) -> np.ndarray:
    q = _c(q, np.uint8)
    out = np.empty(q.shape, np.float64)
    _L().or_e4m3_value_many(_p(q), q.size, _p(out))
    return out


def quant_rows_e4m3(h_bf16, rows: int, d: int):
    """Per-row absmax E4M3 quantisation of bf16 rows -> (uint8 codes [rows*d], f32 scales)."""
    h = _c(h_bf16, np.uint16)
    assert h.size == rows * d
    q = np.empty(rows * d, np.uint8)
    sc = np.empty(rows, np.float32)
    _L().or_quant_rows_e4m3(_p(h), rows, d, _p(q), _p(sc))
    return q, sc


def e2m1_round(x) -> np.ndarray:
    """FP4 E2M1 codes (4-bit, one per byte) of float32 values, nearest-even, saturating."""
    x = _c(x, np.float32)
    out = np.empty(x.size, np.uint8)
    _L().or_e2m1_round_many(_p(x), x.size, _p(out))
    return out


def e2m1_value(q) -> np.ndarray:
    q = _c(q, np.uint8)
    out = np.empty(q.size, np.float64)
    _L().or_e2m1_value_many(_p(q), q.size, _p(out))
    return out


def quant_rows_nvfp4(h_bf16, rows: int, d: int):
    """NVFP4 quantisation of bf16 rows -> (packed E2M1 codes [rows*d/2], E4M3 block scales
    [rows*d/16], fp32 row scales [rows])."""
    h = _c(h_bf16, np.uint16)
    assert h.size == rows * d and d % 16 == 0
    q = np.empty(rows * d // 2, np.uint8)
    bs = np.empty(rows * d // 16, np.uint8)
    sc = np.empty(rows, np.float32)
    _L().or_quant_rows_nvfp4(_p(h), rows, d, _p(q), _p(bs), _p(sc))
    return q, bs, sc


# ---------------------------------------------------------------------------------------------
# one pass
# ---------------------------------------------------------------------------------------------
def head_stats(R: int, d: int, V: int, dtype, h, w, h_scale=None, w_scale=None,
               rows=None, inv_temp: float = 1.0, h_bscale=None, w_bscale=None) -> dict:
    """argmax, conf = max p, entropy H (nats) and the top-2 logit gap for rows of h.
    NVFP4 operands: packed E2M1 codes, per-row fp32 scales and per-16 E4M3 block scales
    [rows][d/16] (h_bscale, w_bscale)."""
    dt = _DT[dtype]
    h = _operand(dt, h)
    w = _operand(dt, w)
    assert _elems(dt, h) == R * d and _elems(dt, w) == V * d
    hb = None if h_bscale is None else _c(h_bscale, np.uint8)
    wb = None if w_bscale is None else _c(w_bscale, np.uint8)
    hs = None if h_scale is None else _c(h_scale, np.float32)
    ws = None if w_scale is None else _c(w_scale, np.float32)
    rr = None if rows is None else _c(rows, np.int64)
    n = R if rr is None else rr.size
    out = {"argmax": np.empty(n, np.int32), "conf": np.empty(n, np.float64),
           "entropy": np.empty(n, np.float64), "gap2": np.empty(n, np.float64)}
    rc = _L().or_head_stats(R, d, V, dt, _p(h), _p(hs), _p(w), _p(ws), float(inv_temp), _p(rr),
                            n, _p(out["argmax"]), _p(out["conf"]), _p(out["entropy"]),
                            _p(out["gap2"]), _p(hb), _p(wb))
    if rc != 0:
        raise RuntimeError(f"or_head_stats failed: {rc}")
    return out


def select(B: int, S: int, V: int, argmax, conf, entropy, keep_k: int, seed: int,
           pass_: int, keep_rule: int = 0, mask_id: int = -1, row_offset: int = 0) -> dict:
    """Mean entropy, top-K keep by (conf desc, slot asc) -- or by (entropy asc, slot asc) with
    keep_rule=1 -- and the new canvas: re-drawn key(seed, pass, row_offset + r) mod V, or mask_id
    when mask_id >= 0 (masked-diffusion variant)."""
    a = _c(argmax, np.int32)
    cf = _c(conf, np.float64)
    en = _c(entropy, np.float64)
    R = B * S
    assert a.size == R and cf.size == R and en.size == R
    out = {"canvas": np.empty(R, np.int32), "kept": np.empty(R, np.uint8),
           "mean_entropy": np.empty(B, np.float64), "kgap": np.empty(B, np.float64)}
    rc = _L().or_select(B, S, V, _p(a), _p(cf), _p(en), int(keep_k), C.c_uint64(seed),
                        C.c_uint32(pass_ & 0xFFFFFFFF), int(keep_rule), int(mask_id),
                        C.c_uint64(row_offset), _p(out["canvas"]), _p(out["kept"]),
                        _p(out["mean_entropy"]), _p(out["kgap"]))
    if rc != 0:
        raise RuntimeError(f"or_select failed: {rc}")
    return out


def step(B: int, S: int, V: int, d: int, dtype, h, w, keep_k: int, seed: int, pass_: int,
         h_scale=None, w_scale=None, inv_temp: float = 1.0, keep_rule: int = 0,
         mask_id: int = -1, row_offset: int = 0, h_bscale=None, w_bscale=None) -> dict:
    """One canvas pass. For an E4M3 or NVFP4 head given bf16 h, h is first quantised per row
    with the head's rule."""
    dt = _DT[dtype]
    out = {}
    if dt == OR_E4M3 and h_scale is None:
        q, sc = quant_rows_e4m3(h, B * S, d)
        h, h_scale = q, sc
        out["q_h"], out["sc_h"] = q, sc
    if dt == OR_NVFP4 and h_scale is None:
        q, bsc, sc = quant_rows_nvfp4(h, B * S, d)
        h, h_bscale, h_scale = q, bsc, sc
        out["q_h"], out["bsc_h"], out["sc_h"] = q, bsc, sc
    st = head_stats(B * S, d, V, dt, h, w, h_scale, w_scale, inv_temp=inv_temp,
                    h_bscale=h_bscale, w_bscale=w_bscale)
    sel = select(B, S, V, st["argmax"], st["conf"], st["entropy"], keep_k, seed, pass_,
                 keep_rule=keep_rule, mask_id=mask_id, row_offset=row_offset)
    out.update(st)
    out.update(sel)
    return out


def synth_denoise(B: int, S: int, d: int, V: int, w_dtype, w, y, canvas, pass_: int,
                  n_content: int, s_content: float, s_pad: float, w_scale=None) -> np.ndarray:
    """Synthetic denoiser h = s * norm(a_t W[y] + (1 - a_t) W[c]), rounded to bf16 bits."""
    dt = _DT[w_dtype]
    w = _operand(dt, w)
    ws = None if w_scale is None else _c(w_scale, np.float32)
    yy = _c(y, np.int32)
    cc = _c(canvas, np.int32)
    h = np.empty(B * S * d, np.uint16)
    rc = _L().or_synth_denoise(B, S, d, V, dt, _p(w), _p(ws), _p(yy), _p(cc),
                               C.c_uint32(pass_), n_content, float(s_content), float(s_pad),
                               _p(h))
    if rc != 0:
        raise RuntimeError(f"or_synth_denoise failed: {rc}")
    return h


# ---------------------------------------------------------------------------------------------
# the denoising loop
# ---------------------------------------------------------------------------------------------
def temperature(p: int, max_passes: int, temp_start: float, temp_end: float) -> float:
    """Sampling temperature of pass p (0-based) on a schedule decaying linearly from temp_start
    at the first pass to temp_end at the last possible pass (0.8 -> 0.4 on the pages:
    "DiffusionGemma 26B: How Google's Text Diffusion Model Generates Tokens in Parallel",
    "Architecture Details"; "When to use a diffusion LLM", "Appendix: Methodology / Decoding")."""
    if max_passes <= 1:
        return float(temp_start)
    return temp_start + (temp_end - temp_start) * p / (max_passes - 1)


def loop(B: int, S: int, V: int, d: int, dtype, w, denoise, *, theta: float,
         stable_passes: int = 2, max_passes: int = 48, keep_k0: int = 32, keep_sched=None,
         seed: int = 0, canvas0=None, start_pass: int = 0, stable0=None, stop_and: bool = False,
         w_scale=None, record: bool = False, temp_start=None, temp_end=None, keep_rule: int = 0,
         mask_id: int = -1, row_offset: int = 0) -> dict:
    """Run the sampler loop; each canvas stops on its own and is frozen after it stops.

    denoise(canvas: int32[R], p: int) -> hidden states for the head: float32 [R*d] for an fp32
    head, bf16 bits [R*d] otherwise (quantised here per row for an E4M3 head).
    Rules after pass p (OR by default; stop_and=True requires entropy AND stability):
      entropy: mean H < theta; stable: canvas unchanged for `stable_passes` consecutive passes;
      cap: p + 1 == max_passes.
    With temp_start/temp_end the statistics of pass p are those of softmax(l / T_p) (see
    temperature()). keep_rule 1 keeps the lowest-entropy slots; mask_id >= 0 is the masked
    variant (the canvas starts all-mask and non-kept slots are re-masked); row_offset shifts the
    rows of the re-draw key (a block's offset in a block-autoregressive run).
    """
    dt = _DT[dtype]
    R = B * S
    if canvas0 is not None:
        c = _c(canvas0, np.int32).copy()
    elif mask_id >= 0:
        c = np.full(R, mask_id, np.int32)
    else:
        c = draw(seed, INIT_PASS, row_offset + np.arange(R, dtype=np.uint64), V)
    stable = np.zeros(B, np.int64) if stable0 is None else np.array(stable0, np.int64)
    done = np.zeros(B, bool)
    passes = np.zeros(B, np.int32)
    reason = np.zeros(B, np.int32)
    last_meanH = np.full(B, np.nan)
    last_argmax = np.zeros(R, np.int32)
    trace = []
    for p in range(start_pass, max_passes):
        t = p + 1
        K = int(keep_sched[p]) if keep_sched is not None else min(keep_k0 * t, S)
        h = denoise(c.copy(), p)
        inv_temp = 1.0 if temp_start is None else 1.0 / temperature(p, max_passes, temp_start,
                                                                   temp_end)
        res = step(B, S, V, d, dt, h, w, K, seed, p, w_scale=w_scale, inv_temp=inv_temp,
                   keep_rule=keep_rule, mask_id=mask_id, row_offset=row_offset)
        if record:
            trace.append({"pass": p, "canvas_in": c.copy(), "h": h, **res})
        for b in range(B):
            if done[b]:
                continue
            sl = slice(b * S, (b + 1) * S)
            changed = bool(np.any(res["canvas"][sl] != c[sl]))
            stable[b] = 0 if changed else stable[b] + 1
            c[sl] = res["canvas"][sl]
            last_meanH[b] = res["mean_entropy"][b]
            last_argmax[sl] = res["argmax"][sl]
            ent = res["mean_entropy"][b] < theta
            stb = stable[b] >= stable_passes
            cap = p + 1 >= max_passes
            stop = ((ent and stb) if stop_and else (ent or stb)) or cap
            if stop:
                done[b] = True
                passes[b] = p + 1
                reason[b] = (REASON_ENTROPY * ent) | (REASON_STABLE * stb) | (REASON_CAP * cap)
        if done.all():
            break
    return {"canvas": c, "passes": passes, "reason": reason, "mean_entropy": last_meanH,
            "argmax": last_argmax, "stable": stable, "trace": trace}


def blocks(n_blocks: int, B: int, S: int, V: int, d: int, dtype, w, y_blocks, *, theta: float,
           n_content: int, s_content: float, s_pad: float, w_scale=None, **loop_kw) -> dict:
    """Block-autoregressive generation with the synthetic denoiser: block i runs the whole
    sampler loop on a fresh canvas with its own targets y_blocks[i] and its re-draw rows offset
    by i*B*S, then commits its final canvas, and block i+1 starts ("DiffusionGemma 26B: How
    Google's Text Diffusion Model Generates Tokens in Parallel", "How Diffusion Changes the
    Equation": the model generates block by block; "When to use a diffusion LLM", "How block
    diffusion works"). Returns the committed tokens [n_blocks*B*S] and per-block passes/reasons."""
    R = B * S
    yb = _c(y_blocks, np.int32).reshape(n_blocks, R)
    tokens = np.empty(n_blocks * R, np.int32)
    passes = np.empty((n_blocks, B), np.int32)
    reason = np.empty((n_blocks, B), np.int32)
    for i in range(n_blocks):
        den = (lambda yy: lambda c, p: synth_denoise(B, S, d, V, dtype, w, yy, c, p, n_content,
                                                     s_content, s_pad, w_scale=w_scale))(yb[i])
        res = loop(B, S, V, d, dtype, w, den, theta=theta, w_scale=w_scale, row_offset=i * R,
                   **loop_kw)
        tokens[i * R:(i + 1) * R] = res["canvas"]
        passes[i], reason[i] = res["passes"], res["reason"]
    return {"tokens": tokens, "passes": passes, "reason": reason}
