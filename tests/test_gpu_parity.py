"""GPU parity: the CUDA path (through the C ABI) against the double-precision oracle on the same
seeded inputs, at sizes spanning several tiles with ragged tails, plus edge cases."""
import numpy as np
import pytest
import torch

from parity import TOL, check_select, check_stats, dev, dev_bf16, dev_u8, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dg():
    from uniform_state_denoising_vocab_b300 import build
    build.build()
    import uniform_state_denoising_vocab_b300 as m
    assert torch.cuda.is_available()
    m.lib()
    return m


def _rand_case(B, S, V, d, seed, dtype, hscale=1.0):
    rng = np.random.default_rng(seed)
    h = (rng.standard_normal(B * S * d) * hscale).astype(np.float32)
    w = (rng.standard_normal(V * d) / np.sqrt(d)).astype(np.float32)
    canvas = rng.integers(0, V, B * S).astype(np.int32)
    return h, w, canvas


def _bits(x):
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _run_step(dg, orc, B, S, V, d, dtype, K, seed, pass_, hscale=1.0, inv_temp=1.0):
    h, w, canvas = _rand_case(B, S, V, d, seed, dtype, hscale)
    if dtype == "f32":
        th, tw = dev(h).view(B * S, d), dev(w).view(V, d)
        oh, ow, ws = h, w, None
        okw = {}
    elif dtype == "bf16":
        hb, wb = _bits(h), _bits(w)
        th, tw = dev_bf16(hb, (B * S, d)), dev_bf16(wb, (V, d))
        oh, ow = hb, wb
        okw = {}
    else:
        hb = _bits(h)
        wq, wsc = orc.quant_rows_e4m3(_bits(w), V, d)
        th, tw = dev_bf16(hb, (B * S, d)), dev_u8(wq, (V, d))
        oh, ow = hb, wq
        okw = {"w_scale": wsc}
    tws = dev(okw["w_scale"]) if "w_scale" in okw else None
    tc = dev(canvas)
    res = dg.dg_canvas_step(th, tw, tc, K, seed, pass_, B=B, S=S, w_scale=tws, inv_temp=inv_temp)
    torch.cuda.synchronize()
    g = {k: host(v) for k, v in res.items() if torch.is_tensor(v)}
    o = orc.step(B, S, V, d, dtype, oh, ow, K, seed, pass_, w_scale=okw.get("w_scale"),
                 inv_temp=inv_temp)
    return g, o, canvas


def test_fp32_pass_v4096_d64(dg, orc):
    """Single canvas pass, fp32 head 4096 x 64, 256 slots, keep 32, seed 0, pass 0."""
    from workloads import CONFIGS, make_pass_inputs
    cfg = CONFIGS["pass_f32_v4096_d64"]
    x = make_pass_inputs(cfg)
    th = dev(x["h"]).view(cfg.R, cfg.d)
    tw = dev(x["w"]).view(cfg.V, cfg.d)
    res = dg.dg_canvas_step(th, tw, dev(x["canvas"]), cfg.keep_k, cfg.seed, 0, B=cfg.B, S=cfg.S)
    torch.cuda.synchronize()
    g = {k: host(v) for k, v in res.items() if torch.is_tensor(v)}
    o = orc.step(cfg.B, cfg.S, cfg.V, cfg.d, "f32", x["h"], x["w"], cfg.keep_k, cfg.seed, 0)
    check_stats(g, o, TOL["f32"])
    check_select(g, o, cfg.B, cfg.S, cfg.V, cfg.keep_k, cfg.seed, 0, orc.draw)
    assert int(g["status"][0]) == 0
    assert abs(g["mean_entropy"][0] - o["mean_entropy"][0]) <= TOL["f32"]


@pytest.mark.parametrize("B,S,V,d", [
    (1, 256, 1000, 128),     # ragged vocabulary tail (3 full tiles + 232)
    (3, 100, 777, 64),       # rows not a multiple of 128; canvases straddle row blocks
    (2, 256, 4096, 256),     # several tiles, several K slices
    (1, 37, 300, 512),       # short canvas
    (1, 256, 256, 64),       # exactly one tile
    (1, 256, 16, 64),        # vocabulary smaller than one 32-column chunk
    (1, 256, 2083, 2816),    # full hidden size, ragged vocabulary
    (1, 256, 1000, 72),      # K tail: the second 64-element slice holds 8 elements (TMA zero fill)
    (2, 150, 2000, 200),     # K tail on the pair kernel (300 rows, two 256-row blocks)
])
def test_bf16_shapes(dg, orc, B, S, V, d):
    g, o, _ = _run_step(dg, orc, B, S, V, d, "bf16", K=min(32, S), seed=V + d, pass_=3)
    check_stats(g, o, TOL["bf16"])
    check_select(g, o, B, S, V, min(32, S), V + d, 3, orc.draw)
    assert int(g["status"][0]) == 0
    assert np.allclose(g["mean_entropy"], o["mean_entropy"], atol=TOL["bf16"])


@pytest.mark.parametrize("B,S,V,d", [(1, 256, 1000, 256), (2, 130, 3001, 2816)])
def test_fp32_shapes(dg, orc, B, S, V, d):
    g, o, _ = _run_step(dg, orc, B, S, V, d, "f32", K=20, seed=5, pass_=1)
    check_stats(g, o, TOL["f32"])
    check_select(g, o, B, S, V, 20, 5, 1, orc.draw)


@pytest.mark.parametrize("B,S,V,d", [(1, 256, 1000, 256), (2, 200, 2500, 2816),
                                     (1, 256, 1000, 208), (1, 100, 700, 48)])  # K tails
def test_e4m3_quantised_head(dg, orc, B, S, V, d):
    g, o, _ = _run_step(dg, orc, B, S, V, d, "e4m3", K=32, seed=11, pass_=0)
    check_stats(g, o, TOL["e4m3"])
    check_select(g, o, B, S, V, 32, 11, 0, orc.draw)


@pytest.mark.parametrize("d", [64, 300])
def test_device_e4m3_quantiser_bit_for_bit(dg, orc, d):
    """dg_quantize_e4m3 (the device's step a0) against the oracle's quantiser code by code:
    rows of wide dynamic range (subnormal codes, saturation at 448), an all-zero row, and rows
    whose products sit exactly on E4M3 midpoints or one fp32 step off them."""
    rng = np.random.default_rng(d)
    R = 40
    x = (rng.standard_normal(R * d) * np.exp(2.5 * rng.standard_normal(R * d))).astype(np.float32)
    x[:d] = 0
    x[d:2 * d] = 0
    x[d:d + 3] = [1.9375, 0.0113525390625, 0.022705078125]
    x[2 * d:3 * d] = 0
    x[2 * d:2 * d + 3] = [3.1875, 0.00933837890625, 0.0186767578125]
    hb = _bits(x)
    got = dg.dg_quantize_e4m3(dev_bf16(hb, (R, d)))
    torch.cuda.synchronize()
    q, sc = orc.quant_rows_e4m3(hb, R, d)
    assert int(got["status"][0]) == 0
    assert np.array_equal(host(got["scale"]), sc)
    gq = host(got["codes"]).reshape(-1)
    zero = lambda c: np.where((c & 0x7F) == 0, 0, c)   # -0 and +0 are the same value
    assert np.array_equal(zero(gq), zero(q))


def test_e4m3_prequantised_h_matches_device_quantiser(dg, orc):
    """bf16 h quantised on the device must give the same statistics, bit for bit, as the
    oracle-quantised E4M3 h passed in directly (the quantiser is exact in fp32)."""
    B, S, V, d = 1, 256, 1500, 512
    h, w, canvas = _rand_case(B, S, V, d, 21, "e4m3")
    hb = _bits(h)
    hq, hsc = orc.quant_rows_e4m3(hb, B * S, d)
    wq, wsc = orc.quant_rows_e4m3(_bits(w), V, d)
    tw, tws = dev_u8(wq, (V, d)), dev(wsc)
    a = dg.dg_canvas_stats(dev_bf16(hb, (B * S, d)), tw, B=B, S=S, w_scale=tws)
    b = dg.dg_canvas_stats(dev_u8(hq, (B * S, d)), tw, B=B, S=S, w_scale=tws, h_scale=dev(hsc))
    torch.cuda.synchronize()
    for k in ("argmax", "conf", "entropy", "mean_entropy"):
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("dtype,B,S,V,d", [
    ("bf16", 1, 256, 30000, 256),     # 118 tiles: more than the pairs, one tile per pair
    ("bf16", 1, 200, 23333, 512),     # 200 rows, ragged vocabulary
    ("bf16", 1, 256, 37888, 2816),    # 148 tiles, 44 K slices through a 3-stage ring
    ("e4m3", 1, 256, 30000, 256),
    ("e4m3", 2, 100, 26000, 2816),
])
def test_pair_head_one_or_two_tiles_per_pair(dg, orc, dtype, B, S, V, d):
    """One 256-row block with more vocabulary tiles than CTA pairs but at most twice as many:
    some pairs take two tiles (both accumulators of a pair in use), the others one."""
    g, o, _ = _run_step(dg, orc, B, S, V, d, dtype, K=32, seed=V % 1000, pass_=1)
    assert int(g["status"][0]) == 0
    check_stats(g, o, TOL[dtype])
    check_select(g, o, B, S, V, 32, V % 1000, 1, orc.draw)


@pytest.mark.parametrize("dtype,V,d", [(dt, V, d) for dt, ds in (("bf16", (8, 16)),
                                                                    ("f32", (4, 8, 16)),
                                                                    ("e4m3", (16,)))
                                         for V in (17, 33, 4097) for d in ds])
def test_tiny_heads(dg, orc, dtype, V, d):
    """The smallest hidden sizes each precision allows (one 16-byte row) and vocabularies just
    past a power of two: one K slice mostly zero-filled, one partial tile."""
    B, S = 2, 130
    g, o, _ = _run_step(dg, orc, B, S, V, d, dtype, K=9, seed=V * d, pass_=4)
    assert int(g["status"][0]) == 0
    check_stats(g, o, TOL[dtype])
    check_select(g, o, B, S, V, 9, V * d, 4, orc.draw)


@pytest.mark.parametrize("dtype,inv_temp", [("bf16", 0.5), ("bf16", 1.25), ("e4m3", 2.5),
                                            ("f32", 0.8)])
def test_inverse_temperature(dg, orc, dtype, inv_temp):
    """The descriptor's inv_temp scales every logit before the statistics (l / T with
    T = 1 / inv_temp): a sharper or flatter softmax, against the oracle at the same scale."""
    B, S, V, d = 2, 150, 2500, 256 if dtype != "f32" else 64
    g, o, _ = _run_step(dg, orc, B, S, V, d, dtype, K=40, seed=17, pass_=2, inv_temp=inv_temp)
    assert int(g["status"][0]) == 0
    check_stats(g, o, TOL[dtype])
    check_select(g, o, B, S, V, 40, 17, 2, orc.draw)


@pytest.mark.parametrize("B,S,K", [(3, 1, 0), (3, 1, 1), (1, 1024, 500), (2, 513, 100)])
def test_canvas_size_extremes(dg, orc, B, S, K):
    """One-slot canvases (each a cluster with seven idle CTAs), the largest canvas the merge
    supports (1024 slots, 128 per CTA of its cluster) and a ragged one."""
    g, o, _ = _run_step(dg, orc, B, S, 3000, 128, "bf16", K=K, seed=S + K, pass_=5)
    check_stats(g, o, TOL["bf16"])
    check_select(g, o, B, S, 3000, K, S + K, 5, orc.draw)
    assert int(g["status"][0]) == 0
    assert np.allclose(g["mean_entropy"], o["mean_entropy"], atol=TOL["bf16"])


@pytest.mark.parametrize("K", [0, 1, 255, 256, 1000])
def test_keep_edges(dg, orc, K):
    g, o, canvas = _run_step(dg, orc, 2, 256, 3000, 128, "bf16", K=K, seed=7, pass_=9)
    check_select(g, o, 2, 256, 3000, K, 7, 9, orc.draw)
    if K == 0:
        assert np.array_equal(g["canvas"], orc.draw(7, 9, np.arange(512), 3000))
    if K >= 256:
        assert np.array_equal(g["canvas"], g["argmax"])


def test_in_place_and_stats_entry_agree(dg, orc):
    B, S, V, d = 1, 256, 5000, 256
    h, w, canvas = _rand_case(B, S, V, d, 3, "bf16")
    th, tw = dev_bf16(_bits(h), (B * S, d)), dev_bf16(_bits(w), (V, d))
    c1 = dev(canvas)
    r1 = dg.dg_canvas_step(th, tw, c1, 32, 1, 2, B=B, S=S)
    c2 = dev(canvas)
    r2 = dg.dg_canvas_step(th, tw, c2, 32, 1, 2, B=B, S=S, canvas_out=c2)   # in place
    st = dg.dg_canvas_stats(th, tw, B=B, S=S)
    torch.cuda.synchronize()
    assert torch.equal(r1["canvas"], c2)
    for k in ("argmax", "conf", "entropy", "mean_entropy"):
        assert torch.equal(r1[k], st[k]) and torch.equal(r1[k], r2[k])


def test_head_clock_sample_is_one_shot(dg):
    """dg_profile_next_head_clock: the next stats call's head writes a plausible SM clock
    sample, later calls leave it alone, and the results are those of an uninstrumented call."""
    B, S, V, d = 1, 256, 20000, 512
    h, w, canvas = _rand_case(B, S, V, d, 6, "bf16")
    th, tw = dev_bf16(_bits(h), (B * S, d)), dev_bf16(_bits(w), (V, d))
    ref = dg.dg_canvas_stats(th, tw, B=B, S=S)
    smp = torch.zeros(4, dtype=torch.int64, device="cuda")
    dg.dg_profile_next_head_clock(smp)
    a = dg.dg_canvas_stats(th, tw, B=B, S=S)
    torch.cuda.synchronize()
    first = smp.clone()
    b = dg.dg_canvas_stats(th, tw, B=B, S=S)
    torch.cuda.synchronize()
    assert torch.equal(smp, first)
    c = host(first).view(np.uint64).astype(np.float64)
    assert c[2] > c[0] and c[3] > c[1]
    assert 200.0 < (c[2] - c[0]) / (c[3] - c[1]) * 1e3 < 2500.0
    for k in ("argmax", "conf", "entropy", "mean_entropy"):
        assert torch.equal(a[k], ref[k]) and torch.equal(b[k], ref[k]), k


def test_deterministic(dg):
    B, S, V, d = 2, 256, 20000, 512
    h, w, canvas = _rand_case(B, S, V, d, 4, "bf16")
    th, tw, tc = dev_bf16(_bits(h), (B * S, d)), dev_bf16(_bits(w), (V, d)), dev(canvas)
    a = dg.dg_canvas_step(th, tw, tc, 40, 9, 4, B=B, S=S)
    b = dg.dg_canvas_step(th, tw, tc, 40, 9, 4, B=B, S=S)
    torch.cuda.synchronize()
    for k in a:
        if torch.is_tensor(a[k]):
            assert torch.equal(a[k], b[k]), k


def test_status_bits(dg):
    B, S, V, d = 1, 256, 1000, 64
    h, w, canvas = _rand_case(B, S, V, d, 5, "bf16")
    th, tw = dev_bf16(_bits(h), (B * S, d)), dev_bf16(_bits(w), (V, d))
    bad = canvas.copy()
    bad[7] = V + 3
    r = dg.dg_canvas_step(th, tw, dev(bad), 8, 0, 0, B=B, S=S)
    torch.cuda.synchronize()
    assert int(r["status"][0]) & dg.ST_BAD_TOKEN
    h2 = h.copy()
    h2[5 * d + 3] = np.nan
    r = dg.dg_canvas_step(dev_bf16(_bits(h2), (B * S, d)), tw, dev(canvas), 8, 0, 0, B=B, S=S)
    torch.cuda.synchronize()
    assert int(r["status"][0]) & dg.ST_NONFINITE
    assert not (int(r["status"][0]) & dg.ST_TIMEOUT)


def test_step_state_and_stop_rule(dg, orc):
    """dg_canvas_step with a state applies the stop test; a stopped canvas is frozen."""
    B, S, V, d = 2, 64, 500, 64
    rng = np.random.default_rng(8)
    w = (rng.standard_normal(V * d) / np.sqrt(d)).astype(np.float32)
    h = (rng.standard_normal(B * S * d) * np.repeat([200.0, 0.05], S * d)).astype(np.float32)
    th, tw = dev_bf16(_bits(h), (B * S, d)), dev_bf16(_bits(w), (V, d))
    state = dg.new_state(B, "cuda")
    rule = dg.StopRule(max_passes=3, entropy_threshold=0.05, stable_passes=2, stop_mode=0)
    c = dev(rng.integers(0, V, B * S).astype(np.int32))
    for p in range(3):
        prev = c.clone()
        dg.dg_canvas_step(th, tw, c, 0, 3, p, B=B, S=S, canvas_out=c, state=state, rule=rule)
        torch.cuda.synchronize()
        f = dg.state_fields(state)
        if p == 0:
            assert f["done"].tolist() == [1, 0] and f["reason"][0] == dg.REASON_ENTROPY
            frozen = c[:S].clone()
        else:
            assert torch.equal(c[:S], frozen)
    f = dg.state_fields(state)
    assert f["passes"].tolist() == [1, 3]
    assert f["reason"][1] == dg.REASON_CAP


@pytest.fixture(scope="module")
def full_pass_inputs():
    from workloads import CONFIGS, make_pass_inputs
    cfg = CONFIGS["pass_bf16_v262144_d2816"]
    return cfg, make_pass_inputs(cfg)


def _full_size_checks(g, o, cfg, tol, draw):
    """Every row of a full-size pass against the oracle (statistics, argmax where pinned), the
    kept set of every canvas against the oracle's (exact where its confidence gap across the
    boundary exceeds 1e-3), the new canvas, the mean entropies, and the size-independent
    properties (entropy in [0, ln V], confidence in [1/V, 1])."""
    check_stats(g, o, tol)
    check_select(g, o, cfg.B, cfg.S, cfg.V, cfg.keep_k, cfg.seed, 0, draw)
    assert int(g["status"][0]) == 0
    assert (g["entropy"] >= 0).all() and (g["entropy"] <= np.log(cfg.V) + 1e-4).all()
    assert (g["conf"] >= 1.0 / cfg.V * 0.999).all() and (g["conf"] <= 1.0).all()
    assert np.allclose(g["mean_entropy"], o["mean_entropy"], atol=tol, rtol=0)
    for b in range(cfg.B):
        sl = slice(b * cfg.S, (b + 1) * cfg.S)
        assert abs(g["mean_entropy"][b] - g["entropy"][sl].astype(np.float64).mean()) < 1e-4


def test_full_vocab_bf16_all_rows(dg, orc, full_pass_inputs):
    """256 slots x 262144 vocab x d=2816 in the launch configuration the benchmark times: every
    row against the oracle, the kept set against the oracle's."""
    cfg, x = full_pass_inputs
    th, tw = dev_bf16(x["h"], (cfg.R, cfg.d)), dev_bf16(x["w"], (cfg.V, cfg.d))
    res = dg.dg_canvas_step(th, tw, dev(x["canvas"]), cfg.keep_k, cfg.seed, 0, B=cfg.B, S=cfg.S)
    torch.cuda.synchronize()
    g = {k: host(v) for k, v in res.items() if torch.is_tensor(v)}
    o = orc.step(cfg.B, cfg.S, cfg.V, cfg.d, "bf16", x["h"], x["w"], cfg.keep_k, cfg.seed, 0)
    _full_size_checks(g, o, cfg, TOL["bf16"], orc.draw)


def test_batched_bf16_all_rows(dg, orc):
    """Eight canvases (2048 rows) x 262144 x 2816: every row, every canvas's kept set and mean
    entropy against the oracle."""
    from workloads import CONFIGS, make_pass_inputs
    cfg = CONFIGS["pass_bf16_b8_v262144_d2816"]
    x = make_pass_inputs(cfg)
    th, tw = dev_bf16(x["h"], (cfg.R, cfg.d)), dev_bf16(x["w"], (cfg.V, cfg.d))
    res = dg.dg_canvas_step(th, tw, dev(x["canvas"]), cfg.keep_k, cfg.seed, 0, B=cfg.B, S=cfg.S)
    torch.cuda.synchronize()
    g = {k: host(v) for k, v in res.items() if torch.is_tensor(v)}
    del th, tw, res
    o = orc.step(cfg.B, cfg.S, cfg.V, cfg.d, "bf16", x["h"], x["w"], cfg.keep_k, cfg.seed, 0)
    _full_size_checks(g, o, cfg, TOL["bf16"], orc.draw)


@pytest.mark.parametrize("V", [1, 2, 3, 255, 65537, 999983])
def test_redraw_modulo_edges(dg, orc, V):
    """With nothing kept every slot is re-drawn: the device's key mod V (computed without the
    64-bit division routine) equals the oracle's plain modulo for small, prime and odd V."""
    B, S, d = 2, 256, 16
    rng = np.random.default_rng(V)
    h = rng.standard_normal(B * S * d).astype(np.float32)
    w = (rng.standard_normal(V * d) / 4).astype(np.float32)
    th, tw = dev_bf16(_bits(h), (B * S, d)), dev_bf16(_bits(w), (V, d))
    canvas = dev(rng.integers(0, V, B * S).astype(np.int32))
    for seed, pass_ in ((0, 0), (12345678901234, 47), (2**64 - 1, 0xFFFFFFFE)):
        r = dg.dg_canvas_step(th, tw, canvas, 0, seed, pass_, B=B, S=S)
        torch.cuda.synchronize()
        assert np.array_equal(host(r["canvas"]), orc.draw(seed, pass_, np.arange(B * S), V))


@pytest.mark.parametrize("keep_rule,mask", [(1, None), (0, 0), (1, 2999)])
def test_keep_rule_and_mask_variants(dg, orc, keep_rule, mask):
    """Lowest-entropy keep and the masked variant (re-mask instead of re-draw) against the
    oracle: statistics in tolerance, the kept set exact where the oracle's key gap across the
    keep boundary exceeds 1e-3, dropped slots exactly the mask id or the counter-hash draw."""
    B, S, V, d, K, seed, p = 2, 200, 3000, 256, 57, 13, 4
    h, w, canvas = _rand_case(B, S, V, d, 31 + keep_rule, "bf16")
    hb, wb = _bits(h), _bits(w)
    res = dg.dg_canvas_step(dev_bf16(hb, (B * S, d)), dev_bf16(wb, (V, d)), dev(canvas), K, seed,
                            p, B=B, S=S, keep_rule=keep_rule, mask_id=mask)
    torch.cuda.synchronize()
    g = {k: host(v) for k, v in res.items() if torch.is_tensor(v)}
    m = -1 if mask is None else mask
    o = orc.step(B, S, V, d, "bf16", hb, wb, K, seed, p, keep_rule=keep_rule, mask_id=m)
    check_stats(g, o, TOL["bf16"])
    check_select(g, o, B, S, V, K, seed, p, orc.draw, keep_rule=keep_rule, mask_id=m)
    key_g = g["conf"].astype(np.float64) if keep_rule == 0 else -g["entropy"].astype(np.float64)
    for b in range(B):
        sl = slice(b * S, (b + 1) * S)
        order = np.lexsort((np.arange(S), -key_g[sl]))
        assert set(np.nonzero(g["kept"][sl])[0]) == set(order[:K])   # the GPU's own ranking
