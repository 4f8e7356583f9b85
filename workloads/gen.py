"""Seeded, chunked, multi-threaded generation of the synthetic canvas workloads.

Every array is a pure function of (seed, domain tag, shape): each chunk of a stream draws from
its own PCG64 generator seeded by ``SeedSequence([seed, tag, chunk])``, so the result does not
depend on the thread count. The arrays stand in for a trained model's hidden states and
vocabulary head: the pages describe a 256-slot canvas over a 262K-token vocabulary
("DiffusionGemma 26B: How Google's Text Diffusion Model Generates Tokens in Parallel",
"Architecture Details"), and no dataset or weights are involved.

Rounding helpers here (bf16 RNE, E4M3 weight quantisation) prepare *inputs* the way a served
checkpoint would store them; they use torch's CPU casts and are not used by the oracle.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

# Domain tags: XOR-free separation of input streams (SeedSequence entropy words).
TAG_H = 0x48    # hidden states h
TAG_W = 0x57    # vocabulary head W
TAG_C = 0x43    # current canvas tokens
TAG_Y = 0x59    # synthetic denoiser targets

_CHUNK = 1 << 22


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def normal_f32(n: int, seed: int, tag: int, std: float = 1.0) -> np.ndarray:
    """n draws of N(0, std^2) as float32 (PCG64 ziggurat per chunk, then scaled in fp32)."""
    out = np.empty(n, dtype=np.float32)
    nch = (n + _CHUNK - 1) // _CHUNK

    def work(i: int) -> None:
        lo, hi = i * _CHUNK, min(n, (i + 1) * _CHUNK)
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tag, i])))
        g.standard_normal(hi - lo, dtype=np.float32, out=out[lo:hi])
        if std != 1.0:
            out[lo:hi] *= np.float32(std)

    if nch <= 1:
        for i in range(nch):
            work(i)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, range(nch)))
    return out


def uniform_ints(n: int, lo: int, hi: int, seed: int, tag: int) -> np.ndarray:
    """n integers uniform in [lo, hi) as int32."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tag, 0])))
    return g.integers(lo, hi, size=n, dtype=np.int64).astype(np.int32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (torch CPU cast, round-to-nearest-even); returns uint16 bits."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bits to float32 exactly."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def quantize_rows_e4m3_bits(w_bf16: np.ndarray, rows: int, d: int) -> tuple[np.ndarray, np.ndarray]:
    """Per-row absmax quantisation of a bf16 weight matrix to FP8-E4M3 (how an FP8 checkpoint
    stores the head): scale = fp32(amax/448), q = e4m3(fp32(w * fp32(448/amax))).

    Returns (uint8 codes [rows*d], float32 scales [rows]). Rows that are all zero get scale 1.
    Chunked over rows to bound memory.
    """
    q = np.empty(rows * d, dtype=np.uint8)
    sc = np.empty(rows, dtype=np.float32)
    step = max(1, (1 << 24) // d)
    wt = torch.from_numpy(np.asarray(w_bf16, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)
    wt = wt.view(rows, d)
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        blk = wt[r0:r1].float()
        amax = blk.abs().amax(dim=1)
        zero = amax == 0
        safe = torch.where(zero, torch.ones_like(amax), amax)
        inv = torch.full_like(safe, 448.0) / safe
        scale = safe / 448.0
        scale[zero] = 1.0
        inv[zero] = 0.0
        codes = (blk * inv[:, None]).to(torch.float8_e4m3fn).view(torch.uint8)
        q[r0 * d:r1 * d] = codes.reshape(-1).numpy()
        sc[r0:r1] = scale.numpy()
    return q, sc


_E2M1_THRESHOLDS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)


def quantize_rows_nvfp4_bits(w_bf16: np.ndarray, rows: int, d: int):
    """NVFP4 quantisation of a bf16 weight matrix (how a 4-bit checkpoint stores the head), in
    float32: g = amax_row / 2688; per block of 16 elements sb = E4M3(bmax / (6 g)) (torch cast,
    nearest-even); codes = E2M1 nearest-even of w / (sb g), saturating at 6 (0 where sb = 0).

    Returns (codes packed two per byte, element 2j in the low nibble [rows*d/2], plain E4M3 block
    scales [rows*d/16], float32 row scales [rows]). Chunked over rows to bound memory.
    """
    assert d % 16 == 0
    q = np.empty(rows * d // 2, dtype=np.uint8)
    bs = np.empty(rows * d // 16, dtype=np.uint8)
    sc = np.empty(rows, dtype=np.float32)
    step = max(1, (1 << 22) // d)
    src = np.asarray(w_bf16, dtype=np.uint16)
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        x = (src[r0 * d:r1 * d].astype(np.uint32) << 16).view(np.float32).reshape(r1 - r0, d)
        ax = np.abs(x)
        amax = ax.max(axis=1)
        zero = amax == 0
        g = np.where(zero, np.float32(1), amax / np.float32(2688)).astype(np.float32)
        g6 = (np.float32(6) * g).astype(np.float32)
        bmax = ax.reshape(r1 - r0, d // 16, 16).max(axis=2)
        t = (bmax / g6[:, None]).astype(np.float32)
        sbt = torch.from_numpy(t).to(torch.float8_e4m3fn)
        sb = sbt.view(torch.uint8).numpy()
        sb[zero] = 0
        sv = sbt.float().numpy()
        sv[zero] = 0
        db = (sv * g[:, None]).astype(np.float32)
        safe = np.where(db > 0, db, np.float32(1))
        y = (x.reshape(r1 - r0, d // 16, 16) / safe[:, :, None]).astype(np.float32)
        a = np.abs(y)
        idx = np.searchsorted(_E2M1_THRESHOLDS, a, side="left")
        tie = (idx < 7) & (a == _E2M1_THRESHOLDS[np.minimum(idx, 6)]) & (idx % 2 == 1)
        code = (idx + tie).astype(np.uint8) | np.where(np.signbit(y), 8, 0).astype(np.uint8)
        code[db == 0] = 0
        code = code.reshape(r1 - r0, d)
        q[r0 * d // 2:r1 * d // 2] = (code[:, 0::2] | (code[:, 1::2] << 4)).reshape(-1)
        bs[r0 * d // 16:r1 * d // 16] = sb.reshape(-1)
        sc[r0:r1] = g
    return q, bs, sc


@dataclass(frozen=True)
class WorkloadConfig:
    """One synthetic workload: B canvases of S slots, hidden size d, vocabulary V."""
    name: str
    precision: str          # "f32" | "bf16" | "e4m3" | "nvfp4"
    B: int
    S: int
    V: int
    d: int
    seed: int
    mode: str               # "pass" | "loop"
    keep_k: int = 32        # pass mode: K; loop mode: k0 in K_t = min(k0*t, S)
    theta: float = 0.05     # loop: mean-entropy stop threshold (nats)
    stable_passes: int = 2
    max_passes: int = 48
    n_content: int = 50
    s_content: float = 8.0
    s_pad: float = 16.0
    note: str = field(default="", compare=False)

    @property
    def R(self) -> int:
        return self.B * self.S


CONFIGS: dict[str, WorkloadConfig] = {
    "pass_f32_v4096_d64": WorkloadConfig(
        "pass_f32_v4096_d64", "f32", 1, 256, 4096, 64, seed=0, mode="pass",
        note="single canvas pass, fp32 head 4096x64"),
    "loop_bf16_v32768_d256": WorkloadConfig(
        "loop_bf16_v32768_d256", "bf16", 1, 256, 32768, 256, seed=0, mode="loop",
        note="full denoise loop, tied bf16 head 32768x256, synthetic denoiser"),
    "pass_bf16_v262144_d2816": WorkloadConfig(
        "pass_bf16_v262144_d2816", "bf16", 1, 256, 262144, 2816, seed=1, mode="pass",
        note="single canvas pass at full vocabulary, bf16 head"),
    "pass_bf16_b8_v262144_d2816": WorkloadConfig(
        "pass_bf16_b8_v262144_d2816", "bf16", 8, 256, 262144, 2816, seed=2, mode="pass",
        note="8 independent canvases (2048 rows), bf16 head"),
    "pass_nvfp4_v262144_d2816": WorkloadConfig(
        "pass_nvfp4_v262144_d2816", "nvfp4", 1, 256, 262144, 2816, seed=4, mode="pass",
        note="single canvas pass, NVFP4 head (E2M1 + per-16 E4M3 block scales + row scale)"),
    "loop_e4m3_v262144_d2816": WorkloadConfig(
        "loop_e4m3_v262144_d2816", "e4m3", 1, 256, 262144, 2816, seed=3, mode="loop",
        note="full denoise loop, FP8-E4M3 head with per-row fp32 scales"),
}


def make_head(cfg: WorkloadConfig, V: int | None = None, d: int | None = None):
    """Vocabulary head W [V, d] ~ N(0, 1/d), stored in the config's precision.

    Returns dict with 'w' (float32 array, or uint16 bf16 bits, or uint8 e4m3 codes) and
    'w_scale' (float32 [V] for e4m3, else None).
    """
    V = cfg.V if V is None else V
    d = cfg.d if d is None else d
    w = normal_f32(V * d, cfg.seed, TAG_W, std=float(1.0 / np.sqrt(d)))
    if cfg.precision == "f32":
        return {"w": w, "w_scale": None}
    wb = f32_to_bf16_bits(w)
    del w
    if cfg.precision == "bf16":
        return {"w": wb, "w_scale": None}
    if cfg.precision == "nvfp4":
        q, bs, sc = quantize_rows_nvfp4_bits(wb, V, d)
        return {"w": q, "w_scale": sc, "w_bscale": bs}
    q, sc = quantize_rows_e4m3_bits(wb, V, d)
    return {"w": q, "w_scale": sc, "w_bf16": wb}


def make_pass_inputs(cfg: WorkloadConfig) -> dict:
    """Inputs of a single canvas pass: h [R, d] ~ N(0,1), W [V, d] ~ N(0,1/d), canvas uniform in [0,V)."""
    R = cfg.R
    h = normal_f32(R * cfg.d, cfg.seed, TAG_H)
    out = make_head(cfg)
    out["h"] = h if cfg.precision == "f32" else f32_to_bf16_bits(h)
    out["canvas"] = uniform_ints(R, 0, cfg.V, cfg.seed, TAG_C)
    return out


def make_loop_inputs(cfg: WorkloadConfig) -> dict:
    """Inputs of the denoising loop: the tied head W and per-canvas targets y.

    y[slot] is uniform in [1, V) for the first n_content slots of each canvas and the PAD id 0
    for the rest (the canvas is always 256 slots and is padded after the answer:
    "When to use a diffusion LLM", "How block diffusion works"). The initial canvas is drawn by
    the sampler itself (uniform-state start), so it is not an input here.
    """
    out = make_head(cfg)
    y = np.zeros(cfg.R, dtype=np.int32)
    for b in range(cfg.B):
        yy = uniform_ints(cfg.n_content, 1, cfg.V, cfg.seed + 1000 * b, TAG_Y)
        y[b * cfg.S: b * cfg.S + cfg.n_content] = yy
    out["y"] = y
    return out
