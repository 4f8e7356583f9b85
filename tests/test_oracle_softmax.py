"""Pins for the oracle's head contraction and softmax statistics (argmax, conf, entropy).

Brute force: exact rational logits (fractions) and a 60-digit softmax with H = -sum p ln p taken
directly (a different formula from the oracle's shifted two-pass form). Closed forms: uniform
logits, two-level logits, the near-one-hot limit. Invariants: bounds and vocabulary permutation.
"""
from fractions import Fraction

import mpmath
import numpy as np
import pytest

mpmath.mp.dps = 60


def _brute(h_vals, w_vals, R, d, V, h_scale=None, w_scale=None):
    """h_vals/w_vals: exact operand values (python floats); returns argmax, conf, H, gap2."""
    out = []
    for r in range(R):
        logits = []
        for n in range(V):
            acc = Fraction(0)
            for k in range(d):
                acc += Fraction(h_vals[r * d + k]) * Fraction(w_vals[n * d + k])
            if h_scale is not None:
                acc *= Fraction(float(h_scale[r])) * Fraction(float(w_scale[n]))
            logits.append(acc)
        m = max(logits)
        a = logits.index(m)
        second = max([x for i, x in enumerate(logits) if i != a], default=None)
        ml = [mpmath.mpf(x.numerator) / x.denominator for x in logits]
        ex = [mpmath.e ** x for x in ml]
        Z = mpmath.fsum(ex)
        p = [e / Z for e in ex]
        H = -mpmath.fsum(pi * mpmath.log(pi) for pi in p if pi > 0)
        gap = float(m - second) if second is not None else np.inf
        out.append((a, float(max(p)), float(H), gap))
    return out


def _bf16_bits(x):
    import torch
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("V,d,R", [(1, 3, 2), (2, 1, 3), (5, 4, 4), (17, 8, 5), (16, 8, 3)])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "e4m3"])
def test_brute_force_small(orc, V, d, R, dtype):
    rng = np.random.default_rng(V * 100 + d * 10 + R)
    h = rng.standard_normal(R * d).astype(np.float32) * np.float32(1.5)
    w = rng.standard_normal(V * d).astype(np.float32)
    hs = ws = None
    if dtype == "f32":
        hv, wv = h.astype(np.float64), w.astype(np.float64)
        ha, wa = h, w
    elif dtype == "bf16":
        ha, wa = _bf16_bits(h), _bf16_bits(w)
        hv = (ha.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        wv = (wa.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    else:
        ha, hs = orc.quant_rows_e4m3(_bf16_bits(h), R, d)
        wa, ws = orc.quant_rows_e4m3(_bf16_bits(w), V, d)
        hv, wv = orc.e4m3_value(ha), orc.e4m3_value(wa)
    got = orc.head_stats(R, d, V, dtype, ha, wa, h_scale=hs, w_scale=ws)
    ref = _brute([float(x) for x in hv], [float(x) for x in wv], R, d, V, hs, ws)
    for r in range(R):
        a, conf, H, gap = ref[r]
        assert got["argmax"][r] == a
        assert abs(got["conf"][r] - conf) < 1e-12
        assert abs(got["entropy"][r] - H) < 1e-12
        if np.isfinite(gap):
            assert abs(got["gap2"][r] - gap) < 1e-12
        else:
            assert not np.isfinite(got["gap2"][r])


def test_brute_force_ties_pick_lowest_index(orc):
    # rows whose logits tie at the maximum: argmax must be the lowest vocabulary index
    V, d = 6, 2
    w = np.array([[0, 0], [1, 0], [0, 1], [1, 0], [0, 1], [0.5, 0.5]], np.float32).reshape(-1)
    h = np.array([[1, 0], [0, 1], [1, 1], [0, 0]], np.float32).reshape(-1)
    got = orc.head_stats(4, d, V, "f32", h, w)
    assert list(got["argmax"]) == [1, 2, 1, 0]
    assert got["gap2"][0] == 0.0 and got["gap2"][1] == 0.0


@pytest.mark.parametrize("V", [1, 17, 4096])
def test_uniform_logits_closed_form(orc, V):
    d, R = 8, 3
    rng = np.random.default_rng(V)
    h = rng.standard_normal(R * d).astype(np.float32)
    w = np.zeros(V * d, np.float32)
    got = orc.head_stats(R, d, V, "f32", h, w)
    assert (got["argmax"] == 0).all()
    assert np.allclose(got["conf"], 1.0 / V, rtol=1e-14, atol=0)
    assert np.allclose(got["entropy"], np.log(V), rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("L", [0.5, 3.0, 20.0, 80.0])
@pytest.mark.parametrize("V", [17, 4096])
def test_two_level_closed_form(orc, L, V):
    # one logit equal to L at vocabulary index j0, every other logit 0
    d, j0 = 4, V // 3
    h = np.array([1.0, 0, 0, 0], np.float32)
    w = np.zeros((V, d), np.float32)
    w[j0, 0] = L
    got = orc.head_stats(1, d, V, "f32", h, w.reshape(-1))
    Z = mpmath.e ** L + (V - 1)
    conf = mpmath.e ** L / Z
    H = mpmath.log(Z) - L * mpmath.e ** L / Z
    assert got["argmax"][0] == j0
    assert abs(got["conf"][0] - float(conf)) <= 1e-12 * float(conf)   # V terms summed: n*eps
    assert abs(got["entropy"][0] - float(H)) <= 1e-12 * float(H) + 1e-300
    if L == 80.0:
        assert got["entropy"][0] < 1e-20


@pytest.mark.parametrize("T", [0.4, 0.8, 2.5])
def test_temperature_closed_forms(orc, T):
    # statistics of softmax(l / T): the two-level closed form with L / T, and uniform logits
    # stay uniform (H = ln V, conf = 1/V) at any temperature
    V, d, j0, L = 1000, 4, 17, 3.0
    h = np.array([1.0, 0, 0, 0], np.float32)
    w = np.zeros((V, d), np.float32)
    w[j0, 0] = L
    got = orc.head_stats(1, d, V, "f32", h, w.reshape(-1), inv_temp=1.0 / T)
    x = mpmath.mpf(L) / mpmath.mpf(T)
    Z = mpmath.e ** x + (V - 1)
    assert got["argmax"][0] == j0
    assert abs(got["conf"][0] - float(mpmath.e ** x / Z)) <= 1e-12
    assert abs(got["entropy"][0] - float(mpmath.log(Z) - x * mpmath.e ** x / Z)) <= 1e-12
    u = orc.head_stats(1, d, V, "f32", h, np.zeros(V * d, np.float32), inv_temp=1.0 / T)
    assert abs(u["entropy"][0] - np.log(V)) <= 1e-12 and abs(u["conf"][0] - 1.0 / V) <= 1e-15


def test_bounds_and_permutation_invariance(orc):
    rng = np.random.default_rng(5)
    R, d, V = 16, 12, 333
    h = (rng.standard_normal(R * d) * 2).astype(np.float32)
    w = rng.standard_normal(V * d).astype(np.float32)
    got = orc.head_stats(R, d, V, "f32", h, w)
    assert (got["entropy"] >= 0).all() and (got["entropy"] <= np.log(V) + 1e-12).all()
    assert (got["conf"] >= 1.0 / V - 1e-15).all() and (got["conf"] <= 1.0).all()
    perm = rng.permutation(V)
    w2 = w.reshape(V, d)[perm].reshape(-1)
    got2 = orc.head_stats(R, d, V, "f32", h, w2)
    inv = np.argsort(perm)
    assert np.array_equal(perm[got2["argmax"]], got["argmax"])
    assert np.allclose(got2["conf"], got["conf"], rtol=1e-12)
    assert np.allclose(got2["entropy"], got["entropy"], rtol=1e-12)
    assert inv.size == V


def test_row_subset_matches_full(orc):
    rng = np.random.default_rng(9)
    R, d, V = 40, 16, 257
    h = rng.standard_normal(R * d).astype(np.float32)
    w = rng.standard_normal(V * d).astype(np.float32)
    full = orc.head_stats(R, d, V, "f32", h, w)
    rows = np.array([39, 0, 17, 17, 5])
    sub = orc.head_stats(R, d, V, "f32", h, w, rows=rows)
    for i, r in enumerate(rows):
        assert sub["argmax"][i] == full["argmax"][r]
        assert sub["conf"][i] == full["conf"][r] and sub["entropy"][i] == full["entropy"][r]


def test_scales_multiply_logits(orc):
    # E4M3 operands with scales equal the f32 head on the dequantised values
    rng = np.random.default_rng(2)
    R, d, V = 4, 32, 50
    hq, hs = orc.quant_rows_e4m3(_bf16_bits(rng.standard_normal(R * d)), R, d)
    wq, ws = orc.quant_rows_e4m3(_bf16_bits(rng.standard_normal(V * d) * 0.2), V, d)
    got = orc.head_stats(R, d, V, "e4m3", hq, wq, h_scale=hs, w_scale=ws)
    # dequantised values are exact in float64 but not float32, so check against brute force
    ref = _brute([float(x) for x in orc.e4m3_value(hq)], [float(x) for x in orc.e4m3_value(wq)],
                 R, d, V, hs, ws)
    for r in range(R):
        assert got["argmax"][r] == ref[r][0]
        assert abs(got["entropy"][r] - ref[r][2]) < 1e-12


@pytest.mark.parametrize("V,d,R", [(1, 16, 2), (5, 16, 3), (17, 32, 4)])
def test_brute_force_small_nvfp4(orc, V, d, R):
    """NVFP4 operands: each element is e2m1(code) * value(block scale) * row scale; the oracle's
    statistics against the exact rational contraction of those values."""
    rng = np.random.default_rng(V * 7 + d + R)
    h = (rng.standard_normal(R * d) * 1.5).astype(np.float32)
    w = rng.standard_normal(V * d).astype(np.float32)
    hq, hb, hs = orc.quant_rows_nvfp4(_bf16_bits(h), R, d)
    wq, wb, ws = orc.quant_rows_nvfp4(_bf16_bits(w), V, d)

    def values(q, b, rows):
        codes = np.stack([q & 0xF, q >> 4], axis=1).reshape(-1)
        return orc.e2m1_value(codes) * orc.e4m3_value(b).repeat(16)

    got = orc.head_stats(R, d, V, "nvfp4", hq, wq, h_scale=hs, w_scale=ws, h_bscale=hb, w_bscale=wb)
    ref = _brute([float(x) for x in values(hq, hb, R)], [float(x) for x in values(wq, wb, V)],
                 R, d, V, hs, ws)
    for r in range(R):
        a, conf, H, gap = ref[r]
        assert got["argmax"][r] == a
        assert abs(got["conf"][r] - conf) < 1e-12
        assert abs(got["entropy"][r] - H) < 1e-12
