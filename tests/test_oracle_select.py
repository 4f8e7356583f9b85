"""Pins for the oracle's keep / re-randomise step and the synthetic denoiser."""
import itertools

import numpy as np
import pytest

M64 = (1 << 64) - 1


def _py_key(seed, p, row):
    def sm(x):
        z = (x + 0x9E3779B97F4A7C15) & M64
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
        return z ^ (z >> 31)
    return sm(sm(sm(seed) ^ p) ^ row)


def _brute_keep(conf, K):
    """Among all size-K subsets, the kept one must dominate: every kept slot beats every
    dropped slot under (conf desc, slot asc). Exactly one subset does; return it."""
    S = len(conf)
    found = []
    for sub in itertools.combinations(range(S), K):
        s = set(sub)
        ok = all((conf[i] > conf[j]) or (conf[i] == conf[j] and i < j)
                 for i in s for j in range(S) if j not in s)
        if ok:
            found.append(s)
    assert len(found) == 1
    return found[0]


@pytest.mark.parametrize("S", [1, 2, 5, 8, 10])
def test_topk_brute_force_with_ties(orc, S):
    rng = np.random.default_rng(S)
    for trial in range(6):
        conf = rng.integers(0, 4, S).astype(np.float64) / 4.0   # many ties
        if trial % 2:
            conf = rng.random(S)
        for K in range(0, S + 2):
            res = orc.select(1, S, 1000, np.arange(S), conf, np.zeros(S), K, 1, 0)
            kept = {i for i in range(S) if res["kept"][i]}
            assert len(kept) == min(K, S)
            if 0 < K < S:
                assert kept == _brute_keep(list(conf), K)


def test_canvas_update_and_mean_entropy(orc):
    B, S, V = 3, 7, 50
    rng = np.random.default_rng(4)
    argmax = rng.integers(0, V, B * S).astype(np.int32)
    conf = rng.random(B * S)
    H = rng.random(B * S) * 3
    seed, p = 99, 5
    res = orc.select(B, S, V, argmax, conf, H, 3, seed, p)
    for b in range(B):
        assert abs(res["mean_entropy"][b] - H[b * S:(b + 1) * S].sum() / S) < 1e-15
        assert res["kept"][b * S:(b + 1) * S].sum() == 3
        order = sorted(range(S), key=lambda j: (-conf[b * S + j], j))
        assert abs(res["kgap"][b] - (conf[b * S + order[2]] - conf[b * S + order[3]])) < 1e-15
    for r in range(B * S):
        want = argmax[r] if res["kept"][r] else _py_key(seed, p, r) % V
        assert res["canvas"][r] == want


def test_kgap_infinite_at_edges(orc):
    S = 4
    for K in (0, 4, 9):
        res = orc.select(1, S, 10, np.zeros(S), np.arange(S) / 10.0, np.zeros(S), K, 0, 0)
        assert np.isinf(res["kgap"][0])


def _bf16v(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)


def test_synth_denoise_mixing_weight(orc):
    # W[y] = e0 and W[c] = e1 (unit rows): h is proportional to (a_t, 1 - a_t) with
    # a_t = min(1, fp32((2 + t)/10)) and t = pass + 1
    d, V = 4, 3
    w = np.zeros((V, d), np.float32)
    w[1, 0] = 1.0
    w[2, 1] = 1.0
    wb = (w.view(np.uint32) >> 16).astype(np.uint16).reshape(-1)
    for p, a in [(0, 0.3), (1, 0.4), (2, 0.5), (6, 0.9), (7, 1.0), (20, 1.0)]:
        h = orc.synth_denoise(1, 1, d, V, "bf16", wb, [1], [2], p, 1, 8.0, 16.0)
        hv = _bf16v(h)
        nrm = np.hypot(a, 1 - a)
        assert abs(hv[0] - 8 * a / nrm) <= 2**-7 * 8 and abs(hv[1] - 8 * (1 - a) / nrm) <= 2**-7 * 8
        assert hv[2] == 0 and hv[3] == 0


def test_synth_denoise_properties(orc):
    rng = np.random.default_rng(8)
    B, S, d, V = 2, 6, 32, 40
    w = (rng.standard_normal(V * d) / np.sqrt(d)).astype(np.float32)
    wb = (w.view(np.uint32) >> 16).astype(np.uint16)
    y = rng.integers(0, V, B * S).astype(np.int32)
    c = rng.integers(0, V, B * S).astype(np.int32)
    h = _bf16v(orc.synth_denoise(B, S, d, V, "bf16", wb, y, c, 3, 2, 8.0, 16.0)).reshape(B * S, d)
    norms = np.linalg.norm(h, axis=1)
    s = np.array([8.0 if (r % S) < 2 else 16.0 for r in range(B * S)])
    assert np.allclose(norms, s, rtol=2**-7)
    # once a_t = 1 the current canvas no longer matters
    h7 = orc.synth_denoise(B, S, d, V, "bf16", wb, y, c, 7, 2, 8.0, 16.0)
    h7b = orc.synth_denoise(B, S, d, V, "bf16", wb, y, (c + 1) % V, 7, 2, 8.0, 16.0)
    assert np.array_equal(h7, h7b)
    # when the canvas already holds the target, h is the scaled unit target row at any pass
    h0 = _bf16v(orc.synth_denoise(B, S, d, V, "bf16", wb, y, y, 0, 2, 8.0, 16.0)).reshape(B * S, d)
    wv = _bf16v(wb).reshape(V, d)
    ref = s[:, None] * wv[y] / np.linalg.norm(wv[y], axis=1)[:, None]
    assert np.allclose(h0, ref, rtol=2**-8, atol=1e-6)
    # zero head rows give h = 0
    hz = orc.synth_denoise(1, 1, d, V, "bf16", np.zeros(V * d, np.uint16), [0], [1], 0, 1, 8, 16)
    assert not hz.any()


def _brute_keep_entropy(H, K):
    """The kept set under (entropy asc, slot asc): every kept slot beats every dropped slot."""
    S = len(H)
    found = [set(sub) for sub in itertools.combinations(range(S), K)
             if all((H[i] < H[j]) or (H[i] == H[j] and i < j)
                    for i in sub for j in range(S) if j not in sub)]
    assert len(found) == 1
    return found[0]


@pytest.mark.parametrize("S", [1, 3, 6, 9])
def test_entropy_keep_brute_force_with_ties(orc, S):
    rng = np.random.default_rng(100 + S)
    for trial in range(5):
        H = rng.integers(0, 3, S).astype(np.float64) / 2.0 if trial % 2 else rng.random(S) * 4
        conf = rng.random(S)    # must be ignored by the entropy rule
        for K in range(0, S + 2):
            res = orc.select(1, S, 777, np.arange(S), conf, H, K, 3, 1, keep_rule=1)
            kept = {i for i in range(S) if res["kept"][i]}
            assert len(kept) == min(K, S)
            if 0 < K < S:
                assert kept == _brute_keep_entropy(list(H), K)
                order = sorted(range(S), key=lambda j: (H[j], j))
                assert abs(res["kgap"][0] - (H[order[K]] - H[order[K - 1]])) < 1e-15


def test_masked_variant_and_row_offset(orc):
    B, S, V = 2, 9, 40
    rng = np.random.default_rng(6)
    argmax = rng.integers(0, V, B * S).astype(np.int32)
    conf, H = rng.random(B * S), rng.random(B * S)
    # re-mask: dropped slots take the mask id, kept slots their argmax
    res = orc.select(B, S, V, argmax, conf, H, 4, 7, 2, mask_id=V - 1)
    assert np.array_equal(res["canvas"], np.where(res["kept"] == 1, argmax, V - 1))
    # a row offset shifts the key's row index: rows r are drawn as key(seed, pass, off + r)
    off = 3 * B * S + 5
    res = orc.select(B, S, V, argmax, conf, H, 4, 7, 2, row_offset=off)
    for r in range(B * S):
        want = argmax[r] if res["kept"][r] else _py_key(7, 2, off + r) % V
        assert res["canvas"][r] == want
    # invalid rules are refused
    with pytest.raises(RuntimeError):
        orc.select(B, S, V, argmax, conf, H, 4, 7, 2, keep_rule=2)
    with pytest.raises(RuntimeError):
        orc.select(B, S, V, argmax, conf, H, 4, 7, 2, mask_id=V)
