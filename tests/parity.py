"""Helpers for GPU-vs-oracle parity tests: device copies of the seeded inputs and the
comparison rules (exact where the decision is pinned by a gap, tolerance otherwise).

Tolerances: entropy and confidence agree within 2e-3 absolute for fp32/bf16 heads and 5e-3
for E4M3 heads; argmax is exact wherever the oracle's top-2 logit gap exceeds 1e-3; the kept
set is exact wherever the oracle's key gap across the keep boundary exceeds 1e-3, and
otherwise may differ only by swaps among slots within 1e-3 of the boundary; re-randomised
tokens are always exact given the kept mask (pure integer hash).

Secondary (stricter) metric, reported and not asserted: the same exactness wherever the gap
exceeds 1e-5 (logits and keys here are of order 1 or larger, so an absolute 1e-5 is at least as
strict as 1e-5 relative). Every check adds to STRICT_REPORT, which the test session prints at
its end (and writes as JSON to the path in DG_PARITY_REPORT, if set): rows and canvases covered
by each rule, and how many of them differ.
"""
import os
from collections import defaultdict

import numpy as np
import torch

GAP = 1e-3
STRICT_GAP = 1e-5
TOL = {"f32": 2e-3, "bf16": 2e-3, "e4m3": 5e-3, "nvfp4": 5e-3}

# test id -> counters
STRICT_REPORT = defaultdict(lambda: defaultdict(int))


def _report():
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    return STRICT_REPORT[test]


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
    strict = o["gap2"] > STRICT_GAP
    rep = _report()
    rep["argmax_rows"] += int(ga.size)
    rep["argmax_rows_gap_gt_1e-3"] += int(pinned.sum())
    rep["argmax_rows_gap_gt_1e-5"] += int(strict.sum())
    rep["argmax_differ_gap_gt_1e-5"] += int((strict & (ga != o["argmax"])).sum())
    rep["argmax_differ_any"] += int((ga != o["argmax"]).sum())
    dc = np.abs(gc.astype(np.float64) - o["conf"])
    dh = np.abs(gh.astype(np.float64) - o["entropy"])
    assert dc.max() <= tol, f"conf max err {dc.max()} at {dc.argmax()}"
    assert dh.max() <= tol, f"entropy max err {dh.max()} at {dh.argmax()}"
    return {"conf_err": float(dc.max()), "entropy_err": float(dh.max()),
            "pinned_frac": float(pinned.mean())}


def check_select(g, o, B, S, V, K, seed, pass_, draw, *, keep_rule=0, mask_id=-1, row_offset=0,
                 canvases=None):
    """g/o: GPU and oracle outputs with kept, canvas, argmax, conf (and entropy for the
    lowest-entropy keep rule); draw = oracle.draw. The oracle's kgap is the gap of its keep key
    across the boundary. mask_id >= 0: dropped slots become mask_id instead of a re-draw.
    canvases: the canvases to check (default all)."""
    R = B * S
    K = max(0, min(K, S))
    kg = g["kept"].astype(bool)
    ko = o["kept"].astype(bool)
    rep = _report()
    okey = o["conf"] if keep_rule == 0 else -np.asarray(o["entropy"], np.float64)
    for b in (range(B) if canvases is None else canvases):
        sl = slice(b * S, (b + 1) * S)
        assert kg[sl].sum() == K, f"canvas {b}: kept {kg[sl].sum()} != {K}"
        rep["kept_canvases"] += 1
        same = np.array_equal(kg[sl], ko[sl])
        if o["kgap"][b] > STRICT_GAP:
            rep["kept_canvases_gap_gt_1e-5"] += 1
            rep["kept_differ_gap_gt_1e-5"] += int(not same)
        if o["kgap"][b] > GAP:
            rep["kept_canvases_gap_gt_1e-3"] += 1
            assert same, f"canvas {b}: kept set differs (gap {o['kgap'][b]})"
        else:
            rep["kept_differ_any"] += int(not same)
            ok = okey[sl]
            order = np.lexsort((np.arange(S), -ok))
            lo = ok[order[K]] if K < S else -np.inf
            hi = ok[order[K - 1]] if K > 0 else np.inf
            diff = np.nonzero(kg[sl] != ko[sl])[0]
            for j in diff:
                assert lo - GAP <= ok[j] <= hi + GAP, f"canvas {b} slot {j} swapped far from boundary"
    rows = row_offset + np.arange(R, dtype=np.uint64)
    dropped = np.full(R, mask_id, np.int32) if mask_id >= 0 else draw(seed, pass_, rows, V)
    expected = np.where(kg, g["argmax"], dropped)
    sel = np.ones(R, bool)
    if canvases is not None:
        sel[:] = False
        for b in canvases:
            sel[b * S:(b + 1) * S] = True
    assert np.array_equal(g["canvas"][sel], expected[sel]), \
        "new canvas != argmax / re-draw under the GPU kept mask"
    agree = sel & (kg == ko) & ((~kg) | (o["gap2"] > GAP))
    assert np.array_equal(g["canvas"][agree], o["canvas"][agree])
