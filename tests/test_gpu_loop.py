"""GPU parity of the whole denoising loop (graph with a conditional WHILE node) against the
oracle: lockstep (the oracle recomputes every pass from the GPU's own canvas and hidden states,
including every stop rule at every pass) and free-run (the oracle runs the loop on its own; the
two runs must agree, or part at a pass where lockstep found a near-tie the tolerance rules
exempt, which is then reported)."""
import numpy as np
import pytest
import torch

from parity import GAP, TOL, _report, check_select, check_stats, dev, dev_bf16, dev_u8, host

pytestmark = pytest.mark.gpu

STOP_MARGIN = 2e-3   # the stop decision may differ where |mean H - theta| is below this


@pytest.fixture(scope="module")
def dg():
    from uniform_state_denoising_vocab_b300 import build
    build.build()
    import uniform_state_denoising_vocab_b300 as m
    m.lib()
    return m


def _bf16_values(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def _gpu_kept(key, S, K):
    """The kept mask the GPU rule implies for its own keys (key desc, slot asc)."""
    B = key.size // S
    kept = np.zeros(key.size, np.uint8)
    for b in range(B):
        c = key[b * S:(b + 1) * S].astype(np.float64)
        order = np.lexsort((np.arange(S), -c))
        kept[b * S + order[:K]] = 1
    return kept


def lockstep(dg, orc, res, *, B, S, V, d, dtype, w, seed, theta, max_passes, stable_passes=2,
             keep=None, keep_k0=32, w_scale=None, stop_and=False, temp=None, keep_rule=0,
             mask_id=-1, row_offset=0, denoise=None):
    """Check every pass the GPU ran against the oracle recomputing it from the GPU's own
    canvas and hidden states:
      - the hidden states against the oracle-side denoiser `denoise(c, p)` (bf16 bits), within
        one bf16 ulp plus the fp32 cancellation error of the synthetic denoiser's mix;
      - statistics within tolerance, argmax exact where the top-2 gap exceeds 1e-3;
      - the kept set against the oracle's (exact where its key gap exceeds 1e-3), the new canvas
        exactly argmax / re-draw under the GPU's kept mask;
      - each canvas's mean entropy, and the whole stop decision at every pass: the entropy rule
        on the GPU's own mean entropy (which must fall on the oracle's side of theta unless they
        are within STOP_MARGIN of it), the stability rule on the canvases the GPU produced, the
        cap; the GPU stops exactly at the first pass where the rule fires, with that reason;
      - canvases that stopped stay frozen.
    Returns {"passes": per-canvas passes, "events": [(pass, argmax diffs, kept diffs, kgap)],
    "stop_exempt": passes whose stop decision was exempt}."""
    R = B * S
    st = dg.state_fields(res["state"])
    passes = st["passes"].numpy().astype(int)
    reason = st["reason"].numpy().astype(int)
    assert (st["done"].numpy() == 1).all()
    P = int(passes.max())
    tc = host(res["trace_canvas"])
    th = host(res["trace_h"].view(torch.int16)).view(np.uint16)
    tm = host(res["trace_mean_entropy"])
    ta, tcf, te = host(res["trace_argmax"]), host(res["trace_conf"]), host(res["trace_entropy"])
    final = host(res["canvas"])
    if mask_id >= 0:
        init = np.full(R, mask_id, np.int32)
    else:
        init = orc.draw(seed, 0xFFFFFFFF, row_offset + np.arange(R, dtype=np.uint64), V)
    assert np.array_equal(tc[0], init)
    stable = np.zeros(B, int)
    events, stop_exempt = [], []
    theta32 = np.float32(theta)
    rng = np.random.default_rng(1234)
    for p in range(P):
        c_p = tc[p]
        c_next = tc[p + 1] if p + 1 < P else final
        hg = th[p].reshape(-1)
        if denoise is not None:
            ho = denoise(c_p, p)
            vg, vo = _bf16_values(hg).astype(np.float64), _bf16_values(ho).astype(np.float64)
            bound = 2.0**-7 * np.maximum(np.abs(vg), np.abs(vo)) + 1e-5
            err = np.abs(vg - vo)
            assert (err <= bound).all(), f"pass {p}: hidden states differ by {err.max()}"
        K = (keep(p) if keep is not None else min(keep_k0 * (p + 1), S))
        inv_temp = 1.0 if temp is None else 1.0 / orc.temperature(p, max_passes, *temp)
        o = orc.step(B, S, V, d, dtype, hg, w, K, seed, p, w_scale=w_scale, inv_temp=inv_temp,
                     keep_rule=keep_rule, mask_id=mask_id, row_offset=row_offset)
        act = [b for b in range(B) if p < passes[b]]
        rows = np.concatenate([np.arange(b * S, (b + 1) * S) for b in act])
        g = {"argmax": ta[p], "conf": tcf[p], "entropy": te[p], "canvas": c_next}
        key = tcf[p] if keep_rule == 0 else -te[p].astype(np.float64)
        g["kept"] = _gpu_kept(key, S, max(0, min(K, S)))
        check_stats(g, {k: o[k][rows] for k in ("argmax", "conf", "entropy", "gap2")},
                    TOL[dtype], rows=rows)
        check_select(g, o, B, S, V, K, seed, p, orc.draw, keep_rule=keep_rule, mask_id=mask_id,
                     row_offset=row_offset, canvases=act)
        nd_a = int((g["argmax"][rows] != o["argmax"][rows]).sum())
        nd_k = int((g["kept"][rows] != o["kept"][rows]).sum())
        if nd_a or nd_k:
            events.append((p, nd_a, nd_k, float(min(o["kgap"][b] for b in act))))
        for b in range(B):
            sl = slice(b * S, (b + 1) * S)
            if p >= passes[b]:
                assert np.array_equal(c_next[sl], c_p[sl]), f"canvas {b} not frozen at pass {p}"
                continue
            assert abs(tm[p][b] - o["mean_entropy"][b]) <= TOL[dtype]
            stable[b] = 0 if np.any(c_next[sl] != c_p[sl]) else stable[b] + 1
            ent = bool(np.float32(tm[p][b]) < theta32)
            if abs(o["mean_entropy"][b] - theta) >= STOP_MARGIN:
                assert ent == bool(o["mean_entropy"][b] < theta), f"pass {p}: entropy rule"
            else:
                stop_exempt.append(p)
            stb = bool(stable[b] >= stable_passes)
            cap = p + 1 >= max_passes
            stop = ((ent and stb) if stop_and else (ent or stb)) or cap
            assert stop == (p + 1 == passes[b]), \
                f"canvas {b} pass {p}: stop {stop} (entropy {ent}, stable {stable[b]}, cap {cap}) " \
                f"but the GPU ran {passes[b]} passes"
            if stop:
                assert reason[b] == (1 if ent else 0) | (2 if stb else 0) | (4 if cap else 0)
    return {"passes": passes, "reason": reason, "events": events, "stop_exempt": stop_exempt,
            "trace_canvas": tc, "final": final}


def free_run(ls, ref, label=""):
    """Compare the GPU's run (lockstep result `ls`) with the oracle's own loop `ref` (run with
    record=True). They must agree on every canvas after every pass, the pass counts, reasons and
    the final canvas, unless they part at a pass where lockstep recorded an exempt near-tie
    (argmax or kept set within the 1e-3 gap rule, or a stop decision within STOP_MARGIN of
    theta): the first such pass is then reported, and the test fails if the parting pass has no
    exempt event."""
    tc, final = ls["trace_canvas"], ls["final"]
    P = int(ls["passes"].max())
    after_g = lambda p: tc[p + 1] if p + 1 < P else final
    tr = ref["trace"]
    after_o = lambda p: tr[p + 1]["canvas_in"] if p + 1 < len(tr) else ref["canvas"]
    part = None
    for p in range(min(P, len(tr))):
        if not np.array_equal(after_g(p), after_o(p)):
            part = p
            break
    rep = _report()
    if part is None and P == len(tr):
        assert list(ls["passes"]) == list(ref["passes"]) and list(ls["reason"]) == list(ref["reason"])
        assert np.array_equal(final, ref["canvas"])
        rep["free_run_identical"] += 1
        return None
    ev_passes = {e[0] for e in ls["events"]}
    if part is None:
        # same canvases over the common passes, different stop pass: only an exempt stop may do that
        q = min(P, len(tr)) - 1
        assert q in ls["stop_exempt"], \
            f"{label}: free run stops differ (GPU {P}, oracle {len(tr)}) with no exempt stop at pass {q}"
        msg = f"{label}: free run parts at the stop decision of pass {q} (mean H within {STOP_MARGIN} of theta)"
    else:
        assert part in ev_passes, f"{label}: free run parts at pass {part} with no near-tie there " \
                                  f"(near-tie events {ls['events']})"
        ev = [e for e in ls["events"] if e[0] == part][0]
        msg = (f"{label}: free run parts at pass {part}: near-tie there ({ev[1]} argmax rows, "
               f"{ev[2]} kept slots within the 1e-3 gap rule, min boundary gap {ev[3]:.2e})")
    rep["free_run_parted_at_exempt_near_tie"] += 1
    print(msg)
    return msg


def _synth(orc, cfg, x, dtype, y=None):
    """Oracle-side synthetic denoiser for a workload (bf16 bits of h for canvas c at pass p)."""
    yy = x["y"] if y is None else y
    return lambda c, p: orc.synth_denoise(cfg.B, cfg.S, cfg.d, cfg.V, dtype, x["w"], yy, c, p,
                                          cfg.n_content, cfg.s_content, cfg.s_pad,
                                          w_scale=x.get("w_scale"))


def _head(cfg, x):
    if cfg.precision == "bf16":
        return dev_bf16(x["w"], (cfg.V, cfg.d)), None
    return dev_u8(x["w"], (cfg.V, cfg.d)), dev(x["w_scale"])


def _run_loop(dg, cfg, x, trace=True, **kw):
    tw, tws = _head(cfg, x)
    canvas = torch.empty(cfg.R, dtype=torch.int32, device="cuda")
    res = dg.dg_canvas_loop(tw, canvas, B=cfg.B, S=cfg.S, theta=cfg.theta, y=dev(x["y"]),
                            w_scale=tws, keep_k0=cfg.keep_k, seed=cfg.seed,
                            max_passes=cfg.max_passes, stable_passes=cfg.stable_passes,
                            n_content=cfg.n_content, s_content=cfg.s_content, s_pad=cfg.s_pad,
                            trace=trace, **kw)
    torch.cuda.synchronize()
    return res


def _loop_checks(dg, orc, cfg, x, res, *, free=True, stop_and=False, **kw):
    """Lockstep every pass, then (free=True) the oracle's own loop against the GPU's run."""
    dtype = cfg.precision
    assert int(res["status"][0]) == 0
    common = dict(B=cfg.B, S=cfg.S, V=cfg.V, d=cfg.d, dtype=dtype, w=x["w"], seed=cfg.seed,
                  theta=cfg.theta, max_passes=cfg.max_passes, stable_passes=cfg.stable_passes,
                  keep_k0=cfg.keep_k, w_scale=x.get("w_scale"), stop_and=stop_and)
    ls = lockstep(dg, orc, res, denoise=_synth(orc, cfg, x, dtype), **common, **kw)
    if not free:
        return ls, None
    okw = {}
    if "temp" in kw:
        okw = dict(temp_start=kw["temp"][0], temp_end=kw["temp"][1])
    for k in ("keep_rule", "mask_id", "row_offset"):
        if k in kw:
            okw[k] = kw[k]
    ref = orc.loop(cfg.B, cfg.S, cfg.V, cfg.d, dtype, x["w"], _synth(orc, cfg, x, dtype),
                   theta=cfg.theta, stable_passes=cfg.stable_passes, max_passes=cfg.max_passes,
                   keep_k0=cfg.keep_k, seed=cfg.seed, w_scale=x.get("w_scale"),
                   stop_and=stop_and, record=True, **okw)
    msg = free_run(ls, ref, cfg.name)
    print(f"{cfg.name}: GPU passes {list(ls['passes'])} reason {list(ls['reason'])}; oracle "
          f"passes {list(ref['passes'])} reason {list(ref['reason'])}; near-tie events "
          f"{ls['events']}; free run: {msg or 'identical'}")
    return ls, ref


def test_loop_bf16_v32768_lockstep_and_free_run(dg, orc):
    from workloads import CONFIGS, make_loop_inputs
    cfg = CONFIGS["loop_bf16_v32768_d256"]
    x = make_loop_inputs(cfg)
    res = _run_loop(dg, cfg, x)
    _loop_checks(dg, orc, cfg, x, res)


def test_loop_e4m3_v32768_lockstep_and_free_run(dg, orc):
    """The FP8 loop at a size the oracle runs in full: E4M3 head with per-row scales, bf16 hidden
    states from the built-in denoiser quantised per row on the device (fused into the denoiser)."""
    from workloads import WorkloadConfig, make_loop_inputs
    cfg = WorkloadConfig("loop_e4m3_v32768_d256", "e4m3", 1, 256, 32768, 256, seed=3, mode="loop")
    x = make_loop_inputs(cfg)
    res = _run_loop(dg, cfg, x)
    _loop_checks(dg, orc, cfg, x, res)


def test_loop_fused_e4m3_quantiser_matches_the_standalone_one(dg, orc):
    """Inside the FP8 loop the built-in denoiser quantises the hidden states it writes (fused);
    quantising the traced bf16 hidden states of each pass with dg_quantize_e4m3 and running the
    same head on them with dg_canvas_stats reproduces that pass's statistics bit for bit, so the
    fused quantiser and the standalone one (checked code by code against the oracle) agree."""
    from workloads import WorkloadConfig, make_loop_inputs
    cfg = WorkloadConfig("loop_e4m3_v32768_d256", "e4m3", 1, 256, 32768, 256, seed=3, mode="loop")
    x = make_loop_inputs(cfg)
    res = _run_loop(dg, cfg, x)
    tw, tws = _head(cfg, x)
    P = int(dg.state_fields(res["state"])["passes"][0])
    assert P >= 2
    for p in range(P):
        q = dg.dg_quantize_e4m3(res["trace_h"][p].view(torch.bfloat16))
        st = dg.dg_canvas_stats(q["codes"], tw, B=cfg.B, S=cfg.S, h_scale=q["scale"],
                                w_scale=tws, h_dtype=dg.DG_E4M3, w_dtype=dg.DG_E4M3)
        torch.cuda.synchronize()
        assert torch.equal(st["argmax"], res["trace_argmax"][p]), p
        assert torch.equal(st["conf"], res["trace_conf"][p]), p
        assert torch.equal(st["entropy"], res["trace_entropy"][p]), p


def test_loop_e4m3_full_scale_lockstep_all_rows(dg, orc):
    """The FP8 loop at 256 slots x 262144 vocab x d=2816 in the launch configuration the
    benchmark times, every pass checked on every row: the denoiser output against the oracle's
    denoiser on the GPU's canvas, all 256 rows' statistics against the oracle (on the GPU's own
    hidden states, quantised by the oracle), the kept set against the oracle's, the new canvas,
    the mean entropy and every stop rule."""
    from workloads import CONFIGS, make_loop_inputs
    cfg = CONFIGS["loop_e4m3_v262144_d2816"]
    x = make_loop_inputs(cfg)
    res = _run_loop(dg, cfg, x)
    ls, _ = _loop_checks(dg, orc, cfg, x, res, free=False)
    P = int(ls["passes"][0])
    assert 1 <= P <= cfg.max_passes
    te, tcf = host(res["trace_entropy"]), host(res["trace_conf"])
    assert (te[:P] >= 0).all() and (te[:P] <= np.log(cfg.V) + 1e-4).all()
    assert (tcf[:P] >= 0.999 / cfg.V).all() and (tcf[:P] <= 1.0).all()
    print(f"full-scale E4M3 loop: {P} passes, reason {int(ls['reason'][0])}, near-tie events "
          f"{ls['events']}")


# The pages give other stop thresholds and an AND combination of the rules: mean entropy below
# 0.005 AND tokens stable ("DiffusionGemma 26B: How Google's Text Diffusion Model Generates Tokens
# in Parallel", "Architecture Details"), entropy_bound = 0.1 ("When to use a diffusion LLM",
# "Appendix: Methodology / Decoding"). Denoiser scales chosen (by running the oracle) so that
# each rule fires mid-loop, away from theta: OR at 0.1 and at 0.005 stop by entropy at pass 6;
# AND at 0.005 and at 0.1 stop at pass 10 with both entropy and stability true, where OR would
# have stopped earlier (pass 1 and pass 6).
STOP_VARIANTS = {
    "or_theta_0.1": dict(theta=0.1, s_content=20.0, s_pad=16.0, stop_and=False, want=(6, 1)),
    "or_theta_0.005": dict(theta=0.005, s_content=24.0, s_pad=20.0, stop_and=False, want=(6, 1)),
    "and_theta_0.005": dict(theta=0.005, s_content=24.0, s_pad=32.0, stop_and=True, want=(10, 3)),
    "and_theta_0.1": dict(theta=0.1, s_content=20.0, s_pad=16.0, stop_and=True, want=(10, 3)),
}


@pytest.mark.parametrize("variant", list(STOP_VARIANTS))
def test_loop_stop_thresholds_and_and_mode(dg, orc, variant):
    """The pages' thresholds (0.005, 0.1) and the AND combination, through the whole loop: every
    pass in lockstep with every stop rule, then the oracle's free run."""
    import dataclasses
    from workloads import CONFIGS, make_loop_inputs
    v = STOP_VARIANTS[variant]
    cfg = dataclasses.replace(CONFIGS["loop_bf16_v32768_d256"], name=f"loop_bf16_{variant}",
                              theta=v["theta"], s_content=v["s_content"], s_pad=v["s_pad"])
    x = make_loop_inputs(cfg)
    res = _run_loop(dg, cfg, x, stop_mode=dg.STOP_AND if v["stop_and"] else dg.STOP_OR)
    ls, ref = _loop_checks(dg, orc, cfg, x, res, stop_and=v["stop_and"])
    # the oracle's own run is the one the scales were chosen for
    assert (int(ref["passes"][0]), int(ref["reason"][0])) == v["want"]


def test_loop_graph_reuse_and_resume(dg):
    """A second call with the same arguments reuses the captured graph and gives the same
    result; resuming from a mid-loop canvas with its stable count reproduces the tail."""
    from workloads import CONFIGS, make_loop_inputs
    cfg = CONFIGS["loop_bf16_v32768_d256"]
    x = make_loop_inputs(cfg)
    tw = dev_bf16(x["w"], (cfg.V, cfg.d))
    ty = dev(x["y"])
    kw = dict(B=cfg.B, S=cfg.S, theta=cfg.theta, y=ty, keep_k0=cfg.keep_k, seed=cfg.seed,
              max_passes=cfg.max_passes, n_content=cfg.n_content, s_content=cfg.s_content,
              s_pad=cfg.s_pad)
    c1 = torch.empty(cfg.R, dtype=torch.int32, device="cuda")
    r1 = dg.dg_canvas_loop(tw, c1, trace=True, **kw)
    torch.cuda.synchronize()
    c1_final = c1.clone()
    s1 = dg.state_fields(r1["state"])
    r2 = dg.dg_canvas_loop(tw, c1, trace=True, **kw)
    torch.cuda.synchronize()
    assert torch.equal(c1, c1_final)
    assert dg.state_fields(r2["state"])["passes"].tolist() == s1["passes"].tolist()
    P = int(s1["passes"][0])
    assert P >= 3
    k = P - 2
    mid = r1["trace_canvas"][k].clone()
    # stable count entering pass k: consecutive unchanged passes before it
    tc = host(r1["trace_canvas"])
    stable = 0
    for p in range(k):
        stable = 0 if np.any(tc[p + 1] != tc[p]) else stable + 1
    state = dg.new_state(cfg.B, "cuda")
    state[0, 2] = stable
    r3 = dg.dg_canvas_loop(tw, mid, init_random=False, start_pass=k, state=state, **kw)
    torch.cuda.synchronize()
    assert torch.equal(mid, c1_final)
    assert dg.state_fields(r3["state"])["passes"].tolist() == s1["passes"].tolist()


def test_prepared_loop_reruns_match_fresh_calls(dg):
    """prepare_loop marshals a loop call once; each run() is a whole loop from a fresh random
    canvas, identical to a dg_canvas_loop call with the same arguments (same canvas, state and
    statistics), run after run."""
    from workloads import CONFIGS, make_loop_inputs
    cfg = CONFIGS["loop_bf16_v32768_d256"]
    x = make_loop_inputs(cfg)
    tw = dev_bf16(x["w"], (cfg.V, cfg.d))
    ty = dev(x["y"])
    kw = dict(B=cfg.B, S=cfg.S, theta=cfg.theta, y=ty, keep_k0=cfg.keep_k, seed=cfg.seed,
              max_passes=cfg.max_passes, n_content=cfg.n_content, s_content=cfg.s_content,
              s_pad=cfg.s_pad)
    c_ref = torch.empty(cfg.R, dtype=torch.int32, device="cuda")
    ref = dg.dg_canvas_loop(tw, c_ref, **kw)
    torch.cuda.synchronize()
    c = torch.empty(cfg.R, dtype=torch.int32, device="cuda")
    loop = dg.prepare_loop(tw, c, **kw)
    for _ in range(3):
        c.fill_(-1)
        out = loop.run()
        torch.cuda.synchronize()
        assert torch.equal(c, c_ref)
        assert torch.equal(out["state"], ref["state"])
        for k in ("argmax", "conf", "entropy"):
            assert torch.equal(out[k], ref[k]), k
        assert int(out["status"][0]) == 0


def test_loop_rules_on_device(dg):
    """Each stop rule fires at the expected pass on the device: cap with nothing kept, entropy
    at the first pass with large logits."""
    V, d, S = 512, 64, 256
    rng = np.random.default_rng(0)
    w = torch.from_numpy((rng.standard_normal((V, d)) / 8).astype(np.float32)).to(torch.bfloat16).cuda()
    y = torch.from_numpy(rng.integers(1, V, S).astype(np.int32)).cuda()
    c = torch.empty(S, dtype=torch.int32, device="cuda")
    # k0 = 0: nothing is ever kept, the canvas changes every pass -> cap at max_passes
    r = dg.dg_canvas_loop(w, c, B=1, S=S, theta=1e-6, y=y, keep_k0=0, seed=3, max_passes=7)
    torch.cuda.synchronize()
    f = dg.state_fields(r["state"])
    assert f["passes"].tolist() == [7] and f["reason"].tolist() == [dg.REASON_CAP]
    # huge scale: every slot one-hot at pass 0 -> entropy rule at the first pass
    r = dg.dg_canvas_loop(w, c, B=1, S=S, theta=0.05, y=y, keep_k0=0, seed=3, s_content=3000.0,
                          s_pad=3000.0, n_content=S)
    torch.cuda.synchronize()
    f = dg.state_fields(r["state"])
    assert f["passes"].tolist() == [1] and f["reason"][0] & dg.REASON_ENTROPY


@pytest.mark.parametrize("dtype,d", [("bf16", 4608), ("e4m3", 8320), ("bf16", 64), ("e4m3", 48)])
def test_denoiser_row_widths(dg, orc, dtype, d):
    """Two loop passes at hidden sizes on both sides of the vectorised denoiser's register limit
    (wider rows take the generic kernel), two canvases of 96 slots: the hidden states within one
    bf16 ulp of the oracle's denoiser, and each pass against the oracle on them."""
    from workloads import WorkloadConfig, make_loop_inputs
    cfg = WorkloadConfig(f"loop_{dtype}_v300_d{d}", dtype, 2, 96, 300, d, seed=9, mode="loop",
                         max_passes=2, n_content=20)
    x = make_loop_inputs(cfg)
    res = _run_loop(dg, cfg, x)
    ls, _ = _loop_checks(dg, orc, cfg, x, res)
    assert ls["passes"].max() >= 1


def test_loop_timeline_trace(dg):
    """The optional per-pass kernel timeline: every pass that ran has ordered denoiser, head and
    merge intervals (each kernel begins after its predecessor began, and ends after it begins);
    passes that did not run stay empty; the loop's results are unchanged by tracing."""
    from workloads import CONFIGS, make_loop_inputs
    cfg = CONFIGS["loop_bf16_v32768_d256"]
    x = make_loop_inputs(cfg)
    tw, ty = dev_bf16(x["w"], (cfg.V, cfg.d)), dev(x["y"])
    kw = dict(B=cfg.B, S=cfg.S, theta=cfg.theta, y=ty, keep_k0=cfg.keep_k, seed=cfg.seed,
              max_passes=cfg.max_passes, n_content=cfg.n_content, s_content=cfg.s_content,
              s_pad=cfg.s_pad)
    c0 = torch.empty(cfg.R, dtype=torch.int32, device="cuda")
    r0 = dg.dg_canvas_loop(tw, c0, **kw)
    c1 = torch.empty(cfg.R, dtype=torch.int32, device="cuda")
    r1 = dg.dg_canvas_loop(tw, c1, timeline=True, sm_clock=True, **kw)
    torch.cuda.synchronize()
    assert torch.equal(c0, c1)
    # each pass that ran has its head's SM clock sample: ordered stamps, a plausible clock, and
    # a global-timer span inside the head's timeline interval; later rows stay zero
    P_ = int(dg.state_fields(r1["state"])["passes"][0])
    ck = host(r1["trace_sm_clock"]).view(np.uint64).astype(np.float64)
    tlr = host(r1["trace_timeline"]).view(np.uint64).reshape(cfg.max_passes, 3, 2)
    for p in range(P_):
        assert ck[p, 2] > ck[p, 0] and ck[p, 3] > ck[p, 1], p
        mhz = (ck[p, 2] - ck[p, 0]) / (ck[p, 3] - ck[p, 1]) * 1e3
        assert 200.0 < mhz < 2500.0, (p, mhz)
        assert tlr[p, 1, 0] <= ck[p, 1] and ck[p, 3] <= tlr[p, 1, 1], p
    assert (ck[P_:] == 0).all()
    st = dg.sm_clock_stats(r1["trace_sm_clock"][:P_])
    assert st["samples"] == P_ and st["head_kcycles"] > 0
    P = int(dg.state_fields(r1["state"])["passes"][0])
    tl = dg.timeline_us(r1["trace_timeline"], cfg.max_passes)
    prev_end = -1.0
    for p in range(P):
        d, h, m = tl[p]["denoise"], tl[p]["head"], tl[p]["merge"]
        assert d is not None and h is not None and m is not None, p
        assert d[0] <= d[1] and h[0] <= h[1] and m[0] <= m[1]
        assert d[0] >= prev_end - 1e-3       # a pass starts after the previous pass ended
        # each kernel gets past its dependency wait only once its predecessor has finished
        assert h[0] >= d[1] - 0.1 and m[0] >= h[1] - 0.1
        prev_end = m[1]
    for p in range(P, cfg.max_passes):
        assert tl[p]["head"] is None and tl[p]["merge"] is None


@pytest.mark.parametrize("variant", ["temperature", "entropy_keep", "masked", "row_offset"])
def test_loop_rule_variants_lockstep(dg, orc, variant):
    """The sampler variants through the whole loop: the 0.8 -> 0.4 temperature schedule,
    lowest-entropy keep, the masked variant (start all-mask, re-mask), and a block's re-draw row
    offset, each checked pass by pass against the oracle (kept set, every stop rule), then
    against the oracle's free run."""
    from workloads import CONFIGS, make_loop_inputs
    cfg = CONFIGS["loop_bf16_v32768_d256"]
    x = make_loop_inputs(cfg)
    if variant == "temperature":
        kw, chk = dict(temp_start=0.8, temp_end=0.4), dict(temp=(0.8, 0.4))
    elif variant == "entropy_keep":
        kw = chk = dict(keep_rule=1)
    elif variant == "masked":
        kw = chk = dict(mask_id=0)
    else:
        kw = chk = dict(row_offset=7 * cfg.R)
    res = _run_loop(dg, cfg, x, **kw)
    ls, _ = _loop_checks(dg, orc, cfg, x, res, **chk)
    assert 1 <= ls["passes"].max() <= cfg.max_passes


def test_block_generate_against_oracle(dg, orc):
    """Block-autoregressive driver, three blocks of the V=32768, d=256 loop workload with
    keep k0 = 32 ("DiffusionGemma 26B: How Google's Text Diffusion Model Generates Tokens in
    Parallel", "How Diffusion Changes the Equation": generation proceeds block by block):
    (1) with one pass and nothing kept, the committed tokens of block i are the oracle's draws
    with rows offset by i*B*S; (2) every block equals a single loop run with that block's
    targets and row offset; each such run is checked in lockstep against the oracle and then
    against the oracle's block driver (oracle.blocks): committed tokens, passes and reasons."""
    import dataclasses
    from workloads import CONFIGS, make_loop_inputs
    cfg = CONFIGS["loop_bf16_v32768_d256"]
    x = make_loop_inputs(cfg)
    n, R = 3, cfg.R
    rng = np.random.default_rng(17)
    yb = np.concatenate([x["y"]] + [np.where(x["y"] > 0, rng.integers(1, cfg.V, R), 0).astype(np.int32)
                                    for _ in range(n - 1)])
    tw, tyb = dev_bf16(x["w"], (cfg.V, cfg.d)), dev(yb)
    base = dict(B=cfg.B, S=cfg.S, theta=cfg.theta, seed=cfg.seed, n_content=cfg.n_content,
                s_content=cfg.s_content, s_pad=cfg.s_pad)
    r1 = dg.dg_block_generate(tw, tyb, n_blocks=n, keep_k0=0, max_passes=1, **base)
    torch.cuda.synchronize()
    assert np.array_equal(host(r1["tokens"]), orc.draw(cfg.seed, 0, np.arange(n * R), cfg.V))
    r2 = dg.dg_block_generate(tw, tyb, n_blocks=n, keep_k0=cfg.keep_k, **base)
    torch.cuda.synchronize()
    assert int(r2["status"][0]) == 0
    tokens = host(r2["tokens"])
    states = host(r2["states"]).reshape(n, cfg.B, 8)
    ref = orc.blocks(n, cfg.B, cfg.S, cfg.V, cfg.d, "bf16", x["w"], yb, theta=cfg.theta,
                     n_content=cfg.n_content, s_content=cfg.s_content, s_pad=cfg.s_pad,
                     keep_k0=cfg.keep_k, seed=cfg.seed, max_passes=cfg.max_passes,
                     stable_passes=cfg.stable_passes)
    for i in range(n):
        yi = yb[i * R:(i + 1) * R]
        c = torch.empty(R, dtype=torch.int32, device="cuda")
        one = dg.dg_canvas_loop(tw, c, y=dev(yi), keep_k0=cfg.keep_k, row_offset=i * R,
                                trace=True, **base)
        torch.cuda.synchronize()
        assert np.array_equal(host(c), tokens[i * R:(i + 1) * R]), f"block {i}"
        assert int(dg.state_fields(one["state"])["passes"][0]) == states[i, 0, 0]
        assert int(dg.state_fields(one["state"])["reason"][0]) == states[i, 0, 1]
        ci = dataclasses.replace(cfg, name=f"block_{i}")
        xi = dict(x, y=yi)
        ls, _ = _loop_checks(dg, orc, ci, xi, one, free=False, row_offset=i * R)
        ref_i = orc.loop(cfg.B, cfg.S, cfg.V, cfg.d, "bf16", x["w"], _synth(orc, cfg, x, "bf16", yi),
                         theta=cfg.theta, keep_k0=cfg.keep_k, seed=cfg.seed,
                         max_passes=cfg.max_passes, stable_passes=cfg.stable_passes,
                         row_offset=i * R, record=True)
        assert np.array_equal(ref_i["canvas"], ref["tokens"][i * R:(i + 1) * R])
        if free_run(ls, ref_i, f"block {i}") is None:
            assert np.array_equal(tokens[i * R:(i + 1) * R], ref["tokens"][i * R:(i + 1) * R])
            assert states[i, 0, 0] == ref["passes"][i][0] and states[i, 0, 1] == ref["reason"][i][0]


def test_caller_denoiser_hook_and_keep_schedule(dg, orc):
    """A caller-supplied dg_denoise_fn (here a ctypes callback that enqueues torch operations on
    the stream it is given, reading the pass index from the device) and a non-linear keep
    schedule K_p = keep_sched[p] (values from 0 to past S), two canvases that stop on their own:
    the hidden states are h_r = E[(c_r + p) mod V] * 2^(p/3 - 2) in bf16 (exact), which the oracle
    restates; every pass is checked in lockstep, then the oracle's free run. Running the prepared
    call again replays the captured loop (the hook is not called again) with equal results."""
    from workloads.gen import bf16_bits_to_f32, f32_to_bf16_bits
    B, S, V, d, maxp, theta, seed = 2, 256, 4096, 64, 24, 1.0, 77
    R = B * S
    rng = np.random.default_rng(41)
    w_bits = f32_to_bf16_bits((rng.standard_normal(V * d) / np.sqrt(d)).astype(np.float32))
    e_bits = f32_to_bf16_bits(rng.standard_normal(V * d).astype(np.float32))
    scale = (2.0 ** (np.arange(maxp) // 3 - 2)).astype(np.float32)
    sched = np.array([0, 3, 300, 17, 64, 1, 255, 256, 0, 128, 40, 200, 7, 99, 256, 31, 2, 180,
                      5, 90, 11, 250, 60, 150], np.int32)
    tw, te = dev_bf16(w_bits, (V, d)), dev_bf16(e_bits, (V, d))
    tsc = torch.from_numpy(scale).to(torch.bfloat16).cuda()
    canvas = torch.empty(R, dtype=torch.int32, device="cuda")
    h_buffer = torch.empty(R, d, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(dg.dg_workspace_bytes(dg.make_desc(h_buffer, tw, B=B, S=S)), dtype=torch.uint8,
                     device="cuda")
    idx = torch.empty(R, dtype=torch.int32, device="cuda")
    sbuf = torch.empty(1, dtype=torch.bfloat16, device="cuda")
    calls, errors = [], []

    def hook(c_ptr, p_ptr, h_ptr, stream):
        try:
            calls.append(1)
            assert c_ptr == canvas.data_ptr() and h_ptr == h_buffer.data_ptr()
            off = p_ptr - ws.data_ptr()
            assert 0 <= off <= ws.numel() - 4 and off % 4 == 0
            pass_t = ws[off:off + 4].view(torch.int32)        # the loop's device pass counter
            with torch.cuda.stream(torch.cuda.ExternalStream(stream)):
                torch.add(canvas, pass_t, out=idx)
                torch.remainder(idx, V, out=idx)
                torch.index_select(te, 0, idx, out=h_buffer)
                torch.index_select(tsc, 0, pass_t, out=sbuf)
                torch.mul(h_buffer, sbuf, out=h_buffer)
            return 0
        except Exception as e:     # a raising ctypes callback would otherwise return garbage
            errors.append(repr(e))
            return 1

    ksched = dev(sched)
    loop = dg.prepare_loop(tw, canvas, B=B, S=S, theta=theta, denoise=hook, h_buffer=h_buffer,
                           workspace=ws, keep_sched=ksched, seed=seed, max_passes=maxp, trace=True)
    res = loop.run()
    torch.cuda.synchronize()
    assert not errors, errors
    assert len(calls) == 1 and int(res["status"][0]) == 0
    first = {k: res[k].clone() for k in ("canvas", "state", "argmax", "conf", "entropy")}

    ef = bf16_bits_to_f32(e_bits).reshape(V, d)

    def oden(c, p):
        return f32_to_bf16_bits((ef[(c.astype(np.int64) + p) % V] * scale[p]).reshape(-1))

    ls = lockstep(dg, orc, res, B=B, S=S, V=V, d=d, dtype="bf16", w=w_bits, seed=seed,
                  theta=theta, max_passes=maxp, keep=lambda p: int(sched[p]), denoise=oden)
    ref = orc.loop(B, S, V, d, "bf16", w_bits, oden, theta=theta, max_passes=maxp,
                   keep_sched=sched, seed=seed, record=True)
    msg = free_run(ls, ref, "caller denoiser")
    assert list(ref["passes"]) == [16, 19] and list(ref["reason"]) == [1, 1]
    print(f"caller denoiser: GPU passes {list(ls['passes'])}; free run: {msg or 'identical'}")
    canvas.fill_(-1)
    again = loop.run()
    torch.cuda.synchronize()
    assert len(calls) == 1, "the cached loop graph should be replayed without the hook"
    for k, v in first.items():
        assert torch.equal(again[k], v), k
