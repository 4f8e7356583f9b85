"""A seeded sweep of random pass shapes over every head precision against the oracle: canvas
count, canvas size, vocabulary, hidden size (multiples of each precision's row-byte rule, often
ending inside a K slice), keep count and pass index drawn at random, the head kernel chosen by
the library for each (single CTA or CTA pair, by row count)."""
import numpy as np
import pytest
import torch

from parity import TOL, check_select, check_stats, dev, dev_bf16, host
from test_gpu_nvfp4 import _nvfp4_case
from test_gpu_parity import _run_step


@pytest.fixture(scope="module")
def dg():
    from uniform_state_denoising_vocab_b300 import build
    build.build()
    import uniform_state_denoising_vocab_b300 as m
    assert torch.cuda.is_available()
    m.lib()
    return m


def _cases(n=16, seed=2026):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        dtype = ("bf16", "e4m3", "f32", "nvfp4")[i % 4]
        B = int(rng.integers(1, 4))
        S = int(rng.integers(1, 301))
        V = int(rng.integers(1, 5001))
        unit = {"bf16": 8, "e4m3": 16, "f32": 4, "nvfp4": 256}[dtype]
        d = unit * int(rng.integers(1, {"bf16": 90, "e4m3": 50, "f32": 40, "nvfp4": 4}[dtype]))
        K = int(rng.integers(0, S + 2))
        out.append((dtype, B, S, V, d, K, int(rng.integers(0, 48))))
    return out


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,B,S,V,d,K,p", _cases())
def test_random_shape_against_oracle(dg, orc, dtype, B, S, V, d, K, p):
    seed = B * 1000003 + S * 1009 + V + d
    if dtype == "nvfp4":
        hb, (wq, wbs, wsc), tw, twb, tws, canvas = _nvfp4_case(dg, B, S, V, d, seed)
        res = dg.dg_canvas_step(dev_bf16(hb, (B * S, d)), tw, dev(canvas), K, seed, p, B=B, S=S,
                                w_scale=tws, w_dtype=dg.DG_NVFP4, w_block_scale=twb)
        torch.cuda.synchronize()
        g = {k: host(v) for k, v in res.items() if torch.is_tensor(v)}
        o = orc.step(B, S, V, d, "nvfp4", hb, wq, K, seed, p, w_scale=wsc, w_bscale=wbs)
        tol = TOL["bf16"]
    else:
        g, o, _ = _run_step(dg, orc, B, S, V, d, dtype, K=K, seed=seed, pass_=p)
        tol = TOL[dtype]
    assert int(g["status"][0]) == 0
    check_stats(g, o, tol)
    check_select(g, o, B, S, V, K, seed, p, orc.draw)
    assert np.allclose(g["mean_entropy"], o["mean_entropy"], atol=tol)
