"""Helpers for GPU-vs-oracle parity tests: device copies of the seeded inputs and the
comparison rules (exact where the decision is pinned by a gap, tolerance otherwise).

Tolerances: entropy and confidence agree within 2e-3 absolute for fp32/bf16 heads and 5e-3
for E4M3 heads; argmax is exact wherever the oracle's top-2 logit gap exceeds 1e-3; the kept
set is exact wherever the oracle's confidence gap across the keep boundary exceeds 1e-3, and
otherwise may differ only by swaps among slots within 1e-3 of the boundary; re-randomised
tokens are always exact given the kept mask (pure integer hash).
"""
import numpy as np
import torch

GAP = 1e-3
TOL = {"f32": 2e-3, "bf16": 2e-3, "e4m3": 5e-3}


def dev_bf16(bits: np.ndarray, shape, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).reshape(shape).to(device)


def dev_u8(codes: np.ndarray, shape, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).reshape(shape).to(device)


def dev(a: np.ndarray, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def host(t):
    return t.detach().cpu().numpy()


def check_stats(g, o, tol, rows=None):
    """g: GPU outputs (numpy) argmax/conf/entropy over all rows; o: oracle over `rows`."""
    ga, gc, gh = g["argmax"], g["conf"], g["entropy"]
    if rows is not None:
        ga, gc, gh = ga[rows], gc[rows], gh[rows]
    pinned = o["gap2"] > GAP
    bad = np.nonzero(pinned & (ga != o["argmax"]))[0]
    assert bad.size == 0, f"argmax mismatch at {bad[:10]} (gaps {o['gap2'][bad[:10]]})"
    dc = np.abs(gc.astype(np.float64) - o["conf"])
    dh = np.abs(gh.astype(np.float64) - o["entropy"])
    assert dc.max() <= tol, f"conf max err {dc.max()} at {dc.argmax()}"
    assert dh.max() <= tol, f"entropy max err {dh.max()} at {dh.argmax()}"
    return {"conf_err": float(dc.max()), "entropy_err": float(dh.max()),
            "pinned_frac": float(pinned.mean())}


def check_select(g, o, B, S, V, K, seed, pass_, draw):
    """g/o: GPU and oracle outputs with kept, canvas, argmax, conf; draw = oracle.draw."""
    R = B * S
    K = max(0, min(K, S))
    kg = g["kept"].astype(bool)
    ko = o["kept"].astype(bool)
    for b in range(B):
        sl = slice(b * S, (b + 1) * S)
        assert kg[sl].sum() == K, f"canvas {b}: kept {kg[sl].sum()} != {K}"
        if o["kgap"][b] > GAP:
            assert np.array_equal(kg[sl], ko[sl]), f"canvas {b}: kept set differs (gap {o['kgap'][b]})"
        else:
            oc = o["conf"][sl]
            order = np.lexsort((np.arange(S), -oc))
            lo = oc[order[K]] if K < S else -np.inf
            hi = oc[order[K - 1]] if K > 0 else np.inf
            diff = np.nonzero(kg[sl] != ko[sl])[0]
            for j in diff:
                assert lo - GAP <= oc[j] <= hi + GAP, f"canvas {b} slot {j} swapped far from boundary"
    draws = draw(seed, pass_, np.arange(R), V)
    expected = np.where(kg, g["argmax"], draws)
    assert np.array_equal(g["canvas"], expected), "new canvas != argmax/hash under the GPU kept mask"
    agree = (kg == ko) & ((~kg) | (o["gap2"] > GAP))
    assert np.array_equal(g["canvas"][agree], o["canvas"][agree])
