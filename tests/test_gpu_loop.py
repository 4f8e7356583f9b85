"""GPU parity of the whole denoising loop (graph with a conditional WHILE node) against the
oracle: lockstep (the oracle recomputes every pass from the GPU's own canvas and hidden states)
and free-run (the oracle runs the loop on its own)."""
import numpy as np
import pytest
import torch

from parity import GAP, TOL, check_select, check_stats, dev, dev_bf16, dev_u8, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dg():
    from uniform_state_denoising_vocab_b300 import build
    build.build()
    import uniform_state_denoising_vocab_b300 as m
    m.lib()
    return m


def _bf16_values(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def _gpu_kept(conf, S, K):
    """The kept mask the GPU rule implies for its own confidences (conf desc, slot asc)."""
    B = conf.size // S
    kept = np.zeros(conf.size, np.uint8)
    for b in range(B):
        c = conf[b * S:(b + 1) * S]
        order = np.lexsort((np.arange(S), -c.astype(np.float64)))
        kept[b * S + order[:K]] = 1
    return kept


def _lockstep(dg, orc, res, cfg, w_host, w_scale_host, y, dtype, rows=None):
    """Check every pass the GPU ran. Returns (number of passes, list of near-tie events)."""
    R, S, V, d = cfg.R, cfg.S, cfg.V, cfg.d
    st = dg.state_fields(res["state"])
    P = int(st["passes"].max())
    tc = host(res["trace_canvas"])
    th = host(res["trace_h"].view(torch.int16)).view(np.uint16)
    tm = host(res["trace_mean_entropy"])
    ta, tcf, te = host(res["trace_argmax"]), host(res["trace_conf"]), host(res["trace_entropy"])
    final = host(res["canvas"])
    events = []
    assert np.array_equal(tc[0], orc.draw(cfg.seed, 0xFFFFFFFF, np.arange(R), V))
    for p in range(P):
        c_p = tc[p]
        c_next = tc[p + 1] if p + 1 < P else final
        # the denoiser output matches the oracle's denoiser on the same canvas within 1 bf16 ulp
        ho = orc.synth_denoise(cfg.B, S, d, V, dtype, w_host, y, c_p, p, cfg.n_content,
                               cfg.s_content, cfg.s_pad, w_scale=w_scale_host)
        hg = th[p].reshape(-1)
        # within one bf16 ulp of the larger magnitude, plus the fp32 cancellation error of the
        # mix a*W[y] + (1-a)*W[c] (about 1e-7 of the terms, times s/|x|): 1e-5 absolute
        vg, vo = _bf16_values(hg).astype(np.float64), _bf16_values(ho).astype(np.float64)
        err = np.abs(vg - vo)
        bound = 2.0**-7 * np.maximum(np.abs(vg), np.abs(vo)) + 1e-5
        assert (err <= bound).all(), f"pass {p}: denoiser differs by {err.max()}"
        K = min(cfg.keep_k * (p + 1), S)
        o = orc.step(cfg.B, S, V, d, dtype, hg, w_host, K, cfg.seed, p, w_scale=w_scale_host)
        g = {"argmax": ta[p], "conf": tcf[p], "entropy": te[p], "canvas": c_next,
             "kept": _gpu_kept(tcf[p], S, K)}
        check_stats(g, o, TOL[dtype])
        check_select(g, o, cfg.B, S, V, K, cfg.seed, p, orc.draw)
        assert abs(tm[p][0] - o["mean_entropy"][0]) <= TOL[dtype]
        if (g["argmax"] != o["argmax"]).any() or (g["kept"] != o["kept"]).any():
            events.append((p, int((g["argmax"] != o["argmax"]).sum()),
                           int((g["kept"] != o["kept"]).sum()), float(o["kgap"][0])))
        # the stop decision at this pass agrees unless the mean entropy is within 2e-3 of theta
        if abs(o["mean_entropy"][0] - cfg.theta) >= 2e-3:
            stopped_here = p + 1 == P
            ent = o["mean_entropy"][0] < cfg.theta
            if ent:
                assert stopped_here
    return P, events


def test_loop_bf16_v32768_lockstep_and_free_run(dg, orc):
    from workloads import CONFIGS, make_loop_inputs
    cfg = CONFIGS["loop_bf16_v32768_d256"]
    x = make_loop_inputs(cfg)
    tw = dev_bf16(x["w"], (cfg.V, cfg.d))
    canvas = torch.empty(cfg.R, dtype=torch.int32, device="cuda")
    res = dg.dg_canvas_loop(tw, canvas, B=cfg.B, S=cfg.S, theta=cfg.theta, y=dev(x["y"]),
                            keep_k0=cfg.keep_k, seed=cfg.seed, max_passes=cfg.max_passes,
                            stable_passes=cfg.stable_passes, n_content=cfg.n_content,
                            s_content=cfg.s_content, s_pad=cfg.s_pad, trace=True)
    torch.cuda.synchronize()
    assert int(res["status"][0]) == 0
    st = dg.state_fields(res["state"])
    assert st["done"][0] == 1
    P, events = _lockstep(dg, orc, res, cfg, x["w"], None, x["y"], "bf16")
    # free run: the oracle's own loop
    den = lambda c, p: orc.synth_denoise(cfg.B, cfg.S, cfg.d, cfg.V, "bf16", x["w"], x["y"], c, p,
                                         cfg.n_content, cfg.s_content, cfg.s_pad)
    ref = orc.loop(cfg.B, cfg.S, cfg.V, cfg.d, "bf16", x["w"], den, theta=cfg.theta,
                   stable_passes=cfg.stable_passes, max_passes=cfg.max_passes,
                   keep_k0=cfg.keep_k, seed=cfg.seed)
    print(f"GPU passes {P} reason {int(st['reason'][0])}; oracle passes {ref['passes'][0]} "
          f"reason {ref['reason'][0]}; near-tie events {events}")
    if not events:
        assert P == ref["passes"][0] and int(st["reason"][0]) == ref["reason"][0]
        assert np.array_equal(host(res["canvas"]), ref["canvas"])


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
    if P >= 3:
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


def _run_loop(dg, cfg, x, trace=True):
    if cfg.precision == "bf16":
        tw, tws = dev_bf16(x["w"], (cfg.V, cfg.d)), None
    else:
        tw, tws = dev_u8(x["w"], (cfg.V, cfg.d)), dev(x["w_scale"])
    canvas = torch.empty(cfg.R, dtype=torch.int32, device="cuda")
    res = dg.dg_canvas_loop(tw, canvas, B=cfg.B, S=cfg.S, theta=cfg.theta, y=dev(x["y"]),
                            w_scale=tws, keep_k0=cfg.keep_k, seed=cfg.seed,
                            max_passes=cfg.max_passes, stable_passes=cfg.stable_passes,
                            n_content=cfg.n_content, s_content=cfg.s_content, s_pad=cfg.s_pad,
                            trace=trace)
    torch.cuda.synchronize()
    return res


def test_loop_e4m3_v32768_lockstep_and_free_run(dg, orc):
    """The FP8 loop at a size the oracle runs in full: E4M3 head with per-row scales, bf16 hidden
    states from the built-in denoiser quantised per row on the device (fused into the denoiser)."""
    from workloads import WorkloadConfig, make_loop_inputs
    cfg = WorkloadConfig("loop_e4m3_v32768_d256", "e4m3", 1, 256, 32768, 256, seed=3, mode="loop")
    x = make_loop_inputs(cfg)
    res = _run_loop(dg, cfg, x)
    assert int(res["status"][0]) == 0
    st = dg.state_fields(res["state"])
    assert st["done"][0] == 1
    P, events = _lockstep(dg, orc, res, cfg, x["w"], x["w_scale"], x["y"], "e4m3")
    den = lambda c, p: orc.synth_denoise(cfg.B, cfg.S, cfg.d, cfg.V, "e4m3", x["w"], x["y"], c, p,
                                         cfg.n_content, cfg.s_content, cfg.s_pad,
                                         w_scale=x["w_scale"])
    ref = orc.loop(cfg.B, cfg.S, cfg.V, cfg.d, "e4m3", x["w"], den, theta=cfg.theta,
                   stable_passes=cfg.stable_passes, max_passes=cfg.max_passes,
                   keep_k0=cfg.keep_k, seed=cfg.seed, w_scale=x["w_scale"])
    print(f"GPU passes {P} reason {int(st['reason'][0])}; oracle passes {ref['passes'][0]} "
          f"reason {ref['reason'][0]}; near-tie events {events}")
    if not events:
        assert P == ref["passes"][0] and int(st["reason"][0]) == ref["reason"][0]
        assert np.array_equal(host(res["canvas"]), ref["canvas"])


def test_loop_e4m3_full_scale_sampled_lockstep(dg, orc):
    """The FP8 loop at 256 slots x 262144 vocab x d=2816 in the launch configuration the
    benchmark times. Every pass: the denoiser output for every row against the oracle's
    denoiser on the GPU's canvas; the statistics of sampled rows against the oracle one by one
    (on the GPU's own hidden states, quantised by the oracle); and, for every row, the
    properties that hold at any size: kept = top-K of the GPU's confidences, the new canvas =
    argmax where kept and the counter hash elsewhere, the mean entropy = mean of the slot
    entropies, entropy in [0, ln V], confidence in [1/V, 1]."""
    from workloads import CONFIGS, make_loop_inputs
    cfg = CONFIGS["loop_e4m3_v262144_d2816"]
    x = make_loop_inputs(cfg)
    res = _run_loop(dg, cfg, x)
    assert int(res["status"][0]) == 0
    st = dg.state_fields(res["state"])
    P = int(st["passes"][0])
    assert st["done"][0] == 1 and 1 <= P <= cfg.max_passes
    R, S, V, d = cfg.R, cfg.S, cfg.V, cfg.d
    tc = host(res["trace_canvas"])
    th = host(res["trace_h"].view(torch.int16)).view(np.uint16)
    tm = host(res["trace_mean_entropy"])
    ta, tcf, te = host(res["trace_argmax"]), host(res["trace_conf"]), host(res["trace_entropy"])
    final = host(res["canvas"])
    assert np.array_equal(tc[0], orc.draw(cfg.seed, 0xFFFFFFFF, np.arange(R), V))
    rng = np.random.default_rng(5)
    stable = 0
    for p in range(P):
        c_p = tc[p]
        c_next = tc[p + 1] if p + 1 < P else final
        ho = orc.synth_denoise(cfg.B, S, d, V, "e4m3", x["w"], x["y"], c_p, p, cfg.n_content,
                               cfg.s_content, cfg.s_pad, w_scale=x["w_scale"])
        vg, vo = _bf16_values(th[p].reshape(-1)).astype(np.float64), _bf16_values(ho).astype(np.float64)
        assert (np.abs(vg - vo) <= 2.0**-7 * np.maximum(np.abs(vg), np.abs(vo)) + 1e-5).all()
        rows = np.sort(rng.choice(R, size=6, replace=False))
        q, sc = orc.quant_rows_e4m3(th[p].reshape(-1), R, d)
        o = orc.head_stats(R, d, V, "e4m3", q, x["w"], h_scale=sc, w_scale=x["w_scale"], rows=rows)
        check_stats({"argmax": ta[p], "conf": tcf[p], "entropy": te[p]}, o, TOL["e4m3"], rows=rows)
        assert (te[p] >= 0).all() and (te[p] <= np.log(V) + 1e-4).all()
        assert (tcf[p] >= 0.999 / V).all() and (tcf[p] <= 1.0).all()
        K = min(cfg.keep_k * (p + 1), S)
        kept = _gpu_kept(tcf[p], S, K).astype(bool)
        expect = np.where(kept, ta[p], orc.draw(cfg.seed, p, np.arange(R), V))
        assert np.array_equal(c_next, expect), f"pass {p}: canvas update"
        assert abs(tm[p][0] - te[p].astype(np.float64).mean()) < 1e-4
        stable = 0 if np.any(c_next != c_p) else stable + 1
        stop = tm[p][0] < cfg.theta or stable >= cfg.stable_passes or p + 1 == cfg.max_passes
        assert stop == (p + 1 == P), f"pass {p}: stop decision"


@pytest.mark.parametrize("dtype,d", [("bf16", 4608), ("e4m3", 8320), ("bf16", 64), ("e4m3", 48)])
def test_denoiser_row_widths(dg, orc, dtype, d):
    """One loop pass at hidden sizes on both sides of the vectorised denoiser's register limit
    (wider rows take the generic kernel): the hidden states within one bf16 ulp of the oracle's
    denoiser, and the pass's statistics and canvas against the oracle on them."""
    from workloads import WorkloadConfig, make_loop_inputs
    cfg = WorkloadConfig(f"loop_{dtype}_v300_d{d}", dtype, 2, 96, 300, d, seed=9, mode="loop",
                         max_passes=2, n_content=20)
    x = make_loop_inputs(cfg)
    res = _run_loop(dg, cfg, x)
    assert int(res["status"][0]) == 0
    P, _ = _lockstep(dg, orc, res, cfg, x["w"], x.get("w_scale"), x["y"], dtype)
    assert P >= 1


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
    r1 = dg.dg_canvas_loop(tw, c1, timeline=True, **kw)
    torch.cuda.synchronize()
    assert torch.equal(c0, c1)
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


def _lockstep_rules(dg, orc, res, cfg, x, dtype, *, temp=None, keep_rule=0, mask_id=-1,
                    row_offset=0):
    """Per-pass check of a loop run with a temperature schedule / keep rule / masked variant /
    row offset: the oracle recomputes each pass from the GPU's own canvas and hidden states."""
    R, S, V, d = cfg.R, cfg.S, cfg.V, cfg.d
    st = dg.state_fields(res["state"])
    P = int(st["passes"].max())
    tc = host(res["trace_canvas"])
    th = host(res["trace_h"].view(torch.int16)).view(np.uint16)
    tm = host(res["trace_mean_entropy"])
    ta, tcf, te = host(res["trace_argmax"]), host(res["trace_conf"]), host(res["trace_entropy"])
    final = host(res["canvas"])
    init = (np.full(R, mask_id, np.int32) if mask_id >= 0
            else orc.draw(cfg.seed, 0xFFFFFFFF, row_offset + np.arange(R, dtype=np.uint64), V))
    assert np.array_equal(tc[0], init)
    for p in range(P):
        c_next = tc[p + 1] if p + 1 < P else final
        inv_temp = 1.0 if temp is None else 1.0 / orc.temperature(p, cfg.max_passes, *temp)
        K = min(cfg.keep_k * (p + 1), S)
        o = orc.step(cfg.B, S, V, d, dtype, th[p].reshape(-1), x["w"], K, cfg.seed, p,
                     w_scale=x.get("w_scale"), inv_temp=inv_temp, keep_rule=keep_rule,
                     mask_id=mask_id, row_offset=row_offset)
        check_stats({"argmax": ta[p], "conf": tcf[p], "entropy": te[p]}, o, TOL[dtype])
        assert abs(tm[p][0] - o["mean_entropy"][0]) <= TOL[dtype]
        key = tcf[p].astype(np.float64) if keep_rule == 0 else -te[p].astype(np.float64)
        kept = _gpu_kept(key, S, K).astype(bool)
        dropped = (np.full(R, mask_id) if mask_id >= 0 else
                   orc.draw(cfg.seed, p, row_offset + np.arange(R, dtype=np.uint64), V))
        assert np.array_equal(c_next, np.where(kept, ta[p], dropped)), f"pass {p}"
    return P


@pytest.mark.parametrize("variant", ["temperature", "entropy_keep", "masked", "row_offset"])
def test_loop_rule_variants_lockstep(dg, orc, variant):
    """The NEXT-row sampler variants through the whole loop: the 0.8 -> 0.4 temperature
    schedule, lowest-entropy keep, the masked variant (start all-mask, re-mask), and a block's
    re-draw row offset, each checked pass by pass against the oracle."""
    from workloads import CONFIGS, make_loop_inputs
    cfg = CONFIGS["loop_bf16_v32768_d256"]
    x = make_loop_inputs(cfg)
    kw = {}
    chk = {}
    if variant == "temperature":
        kw = dict(temp_start=0.8, temp_end=0.4)
        chk = dict(temp=(0.8, 0.4))
    elif variant == "entropy_keep":
        kw = chk = dict(keep_rule=1)
    elif variant == "masked":
        kw = dict(mask_id=0)
        chk = dict(mask_id=0)
    else:
        kw = chk = dict(row_offset=7 * cfg.R)
    tw = dev_bf16(x["w"], (cfg.V, cfg.d))
    canvas = torch.empty(cfg.R, dtype=torch.int32, device="cuda")
    res = dg.dg_canvas_loop(tw, canvas, B=cfg.B, S=cfg.S, theta=cfg.theta, y=dev(x["y"]),
                            keep_k0=cfg.keep_k, seed=cfg.seed, max_passes=cfg.max_passes,
                            stable_passes=cfg.stable_passes, n_content=cfg.n_content,
                            s_content=cfg.s_content, s_pad=cfg.s_pad, trace=True, **kw)
    torch.cuda.synchronize()
    assert int(res["status"][0]) == 0
    P = _lockstep_rules(dg, orc, res, cfg, x, "bf16", **chk)
    assert 1 <= P <= cfg.max_passes


def test_block_generate(dg, orc):
    """Block-autoregressive driver: (1) with one pass and nothing kept, the committed tokens of
    block i are the oracle's draws with rows offset by i*B*S; (2) every block equals a single
    loop run with that block's targets and row offset (one captured graph serves all blocks)."""
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
    states = host(r2["states"]).reshape(n, cfg.B, 8)
    for i in range(n):
        c = torch.empty(R, dtype=torch.int32, device="cuda")
        one = dg.dg_canvas_loop(tw, c, y=dev(yb[i * R:(i + 1) * R]), keep_k0=cfg.keep_k,
                                row_offset=i * R, **base)
        torch.cuda.synchronize()
        assert torch.equal(c, r2["tokens"][i * R:(i + 1) * R]), f"block {i}"
        assert int(dg.state_fields(one["state"])["passes"][0]) == states[i, 0, 0]
