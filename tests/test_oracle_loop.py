"""Pins for the oracle's loop control: each stop rule fires at a known pass, the first
qualifying pass ends the loop, canvases in a batch stop independently, and resume is exact."""
import numpy as np
import pytest


def _bf16(x):
    import torch
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


B, S, V, d = 1, 16, 64, 8


@pytest.fixture(scope="module")
def head():
    rng = np.random.default_rng(12)
    return _bf16(rng.standard_normal(V * d) / np.sqrt(d))


def _const_h(scale, R=B * S, seed=3):
    rng = np.random.default_rng(seed)
    return _bf16(rng.standard_normal(R * d) * scale)


def test_entropy_rule_first_pass(orc, head):
    h = _const_h(4000.0)          # huge logits: every slot near one-hot
    res = orc.loop(B, S, V, d, "bf16", head, lambda c, p: h, theta=0.05, keep_k0=0, seed=1)
    assert res["passes"][0] == 1 and res["reason"][0] & 1
    assert res["mean_entropy"][0] < 0.05


def test_stability_rule(orc, head):
    h = _const_h(1.0)
    st = orc.step(B, S, V, d, "bf16", h, head, S, 0, 0)
    # canvas already equal to the argmax: pass 0 and pass 1 both leave it unchanged
    res = orc.loop(B, S, V, d, "bf16", head, lambda c, p: h, theta=1e-9, keep_k0=S, seed=1,
                   canvas0=st["argmax"])
    assert res["passes"][0] == 2 and res["reason"][0] == 2
    # from a random canvas the first pass changes it, so the rule fires one pass later
    res = orc.loop(B, S, V, d, "bf16", head, lambda c, p: h, theta=1e-9, keep_k0=S, seed=1)
    assert res["passes"][0] == 3 and res["reason"][0] == 2
    assert np.array_equal(res["canvas"], st["argmax"])
    # stable_passes = 1 reading: stop at the first pass that changes nothing
    res = orc.loop(B, S, V, d, "bf16", head, lambda c, p: h, theta=1e-9, keep_k0=S, seed=1,
                   stable_passes=1)
    assert res["passes"][0] == 2


def test_cap_rule(orc, head):
    h = _const_h(0.01)           # near-uniform predictions, high entropy
    res = orc.loop(B, S, V, d, "bf16", head, lambda c, p: h, theta=0.05, keep_k0=0, seed=2)
    assert res["passes"][0] == 48 and res["reason"][0] == 4
    res = orc.loop(B, S, V, d, "bf16", head, lambda c, p: h, theta=0.05, keep_k0=0, seed=2,
                   max_passes=5)
    assert res["passes"][0] == 5 and res["reason"][0] == 4


def test_first_qualifying_pass_and_schedule(orc, head):
    # the scale of h grows with the pass, so mean entropy falls below theta at some pass p*;
    # the loop must stop exactly there.
    base = np.random.default_rng(4).standard_normal(B * S * d)
    den = lambda c, p: _bf16(base * (0.5 + 3.0 * p))
    meanH = []
    for p in range(48):
        st = orc.step(B, S, V, d, "bf16", den(None, p), head, 0, 0, p)
        meanH.append(st["mean_entropy"][0])
    theta = 0.2
    pstar = next(p for p, m in enumerate(meanH) if m < theta)
    assert 1 <= pstar < 47
    res = orc.loop(B, S, V, d, "bf16", head, den, theta=theta, keep_k0=0, seed=5)
    assert res["passes"][0] == pstar + 1 and res["reason"][0] & 1


def test_keep_schedule_counts(orc, head):
    # K_t = min(k0 * t, S) with t = pass + 1: record the kept count per pass
    h = _const_h(0.3)
    res = orc.loop(B, S, V, d, "bf16", head, lambda c, p: h, theta=0.0, keep_k0=3, seed=7,
                   max_passes=8, record=True)
    counts = [int(tr["kept"].sum()) for tr in res["trace"]]
    assert counts[: len(counts)] == [min(3 * (p + 1), S) for p in range(len(counts))]


def test_and_mode(orc, head):
    h = _const_h(4000.0)
    st = orc.step(B, S, V, d, "bf16", h, head, S, 0, 0)
    res = orc.loop(B, S, V, d, "bf16", head, lambda c, p: h, theta=0.05, keep_k0=S, seed=1,
                   stop_and=True)
    # entropy holds from pass 0, stability needs two unchanged passes after the first change
    assert res["passes"][0] == 3 and res["reason"][0] == 3
    res = orc.loop(B, S, V, d, "bf16", head, lambda c, p: h, theta=0.05, keep_k0=S, seed=1,
                   stop_and=True, canvas0=st["argmax"])
    assert res["passes"][0] == 2


def test_batch_canvases_stop_independently(orc, head):
    B2 = 2
    rng = np.random.default_rng(6)
    hs = rng.standard_normal(B2 * S * d)
    scale = np.concatenate([np.full(S * d, 4000.0), np.full(S * d, 0.01)])
    h = _bf16(hs * scale)
    res = orc.loop(B2, S, V, d, "bf16", head, lambda c, p: h, theta=0.05, keep_k0=0, seed=3,
                   max_passes=6, record=True)
    assert list(res["passes"]) == [1, 6]
    assert list(res["reason"]) == [1, 4]
    # canvas 0 is frozen after pass 0
    first = res["trace"][0]["canvas"][:S]
    assert np.array_equal(res["canvas"][:S], first)


def test_resume_matches_straight_run(orc, head):
    base = np.random.default_rng(9).standard_normal(B * S * d)
    den = lambda c, p: _bf16(base * 0.7 + np.sin(np.arange(B * S * d) * 0.1 * (p + 1)))
    full = orc.loop(B, S, V, d, "bf16", head, den, theta=0.0, keep_k0=2, seed=4, max_passes=12,
                    record=True)
    k = 5
    mid = full["trace"][k]["canvas_in"]
    # stable count entering pass k, recomputed from the trace
    stable = 0
    for tr in full["trace"][:k]:
        stable = 0 if np.any(tr["canvas"] != tr["canvas_in"]) else stable + 1
    res = orc.loop(B, S, V, d, "bf16", head, den, theta=0.0, keep_k0=2, seed=4, max_passes=12,
                   canvas0=mid, start_pass=k, stable0=[stable])
    assert np.array_equal(res["canvas"], full["canvas"])
    assert list(res["passes"]) == list(full["passes"])


def test_temperature_schedule_per_pass(orc):
    """With a temperature schedule the statistics of pass p are those of softmax(l / T_p),
    T_p falling linearly from 0.8 at the first pass to 0.4 at the last possible pass: every slot
    has two-level logits (L at one id, 0 elsewhere), so each pass's mean entropy is the closed
    form at T_p."""
    import mpmath
    Vt, dt, St, L, P = 50, 8, 4, 2.0, 6
    w = np.zeros((Vt, dt), np.float32)
    w[7, 0] = 1.0
    wb = _bf16(w.reshape(-1))
    h = _bf16(np.tile(np.array([L] + [0.0] * (dt - 1), np.float32), St))
    assert orc.temperature(0, P, 0.8, 0.4) == 0.8 and abs(orc.temperature(P - 1, P, 0.8, 0.4) - 0.4) < 1e-15
    res = orc.loop(1, St, Vt, dt, "bf16", wb, lambda c, p: h, theta=1e-9, keep_k0=0, seed=4,
                   max_passes=P, temp_start=0.8, temp_end=0.4, record=True)
    assert res["passes"][0] == P
    for tr in res["trace"]:
        T = 0.8 - 0.4 * tr["pass"] / (P - 1)
        x = mpmath.mpf(L) / T
        Z = mpmath.e ** x + (Vt - 1)
        H = float(mpmath.log(Z) - x * mpmath.e ** x / Z)
        assert abs(tr["mean_entropy"][0] - H) < 1e-12
        assert (tr["argmax"] == 7).all()


def test_masked_variant_loop(orc, head):
    """Masked variant: the canvas starts all-mask, and a pass keeping every slot sets every slot
    to its argmax; with nothing kept the canvas stays all-mask and the loop ends by stability."""
    mask = V - 1
    h = _const_h(1.0)
    st = orc.step(B, S, V, d, "bf16", h, head, S, 0, 0)
    res = orc.loop(B, S, V, d, "bf16", head, lambda c, p: h, theta=1e-9, keep_k0=S, seed=1,
                   mask_id=mask, record=True)
    assert (res["trace"][0]["canvas_in"] == mask).all()
    assert np.array_equal(res["canvas"], st["argmax"])
    res = orc.loop(B, S, V, d, "bf16", head, lambda c, p: h, theta=1e-9, keep_k0=0, seed=1,
                   mask_id=mask)
    assert (res["canvas"] == mask).all() and res["passes"][0] == 2 and res["reason"][0] == 2


def test_row_offset_initial_canvas(orc, head):
    """A block's row offset shifts the rows of the initial random canvas's key as well."""
    from test_oracle_select import _py_key
    h = _const_h(0.01)
    off = 5 * B * S
    res = orc.loop(B, S, V, d, "bf16", head, lambda c, p: h, theta=0.05, keep_k0=0, seed=2,
                   max_passes=1, row_offset=off, record=True)
    want = [_py_key(2, 0xFFFFFFFF, off + r) % V for r in range(B * S)]
    assert list(res["trace"][0]["canvas_in"]) == want


def test_block_driver_offsets(orc, head):
    """Block i of a block-autoregressive run keys its draws with rows offset by i*B*S: with one
    pass and nothing kept, every committed token of block i is key(seed, 0, i*B*S + r) mod V
    (independent Python restatement of the key); and block i equals a single loop with that
    offset and block i's targets."""
    from test_oracle_select import _py_key
    n, R = 3, B * S
    rng = np.random.default_rng(21)
    yb = rng.integers(0, V, n * R).astype(np.int32)
    kw = dict(theta=0.05, n_content=5, s_content=8.0, s_pad=16.0)
    res = orc.blocks(n, B, S, V, d, "bf16", head, yb, keep_k0=0, seed=9, max_passes=1, **kw)
    assert list(res["tokens"]) == [_py_key(9, 0, r) % V for r in range(n * R)]
    res = orc.blocks(n, B, S, V, d, "bf16", head, yb, keep_k0=4, seed=9, **kw)
    for i in range(n):
        den = lambda c, p, yy=yb[i * R:(i + 1) * R]: orc.synth_denoise(B, S, d, V, "bf16", head, yy,
                                                                    c, p, 5, 8.0, 16.0)
        one = orc.loop(B, S, V, d, "bf16", head, den, theta=0.05, keep_k0=4, seed=9, row_offset=i * R)
        assert np.array_equal(res["tokens"][i * R:(i + 1) * R], one["canvas"])
        assert res["passes"][i][0] == one["passes"][0]
