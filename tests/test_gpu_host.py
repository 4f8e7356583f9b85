"""dg_canvas_step_host: the canvas pass on host buffers gives exactly the results of
dg_canvas_step on device copies of the same inputs, call after call (the two staging sets
alternate and each call's uploads overlap the previous call's kernels)."""
import numpy as np
import pytest
import torch

from parity import dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dg():
    from uniform_state_denoising_vocab_b300 import build
    build.build()
    import uniform_state_denoising_vocab_b300 as m
    m.lib()
    return m


def _bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _case(dg, precision, B, S, V, d, seed):
    """Device head, device h operand(s) and the matching descriptor keywords."""
    rng = np.random.default_rng(seed)
    hb = _bits(rng.standard_normal(B * S * d))
    wb = _bits(rng.standard_normal(V * d) / np.sqrt(d))
    th = dev_bf16(hb, (B * S, d))
    tw = dev_bf16(wb, (V, d))
    if precision == "bf16":
        return {"h": th}, tw, {}
    if precision == "e4m3":
        wq = tw.float()
        wsc = wq.abs().amax(1).clamp_min(1e-30) / 448.0
        w8 = (wq / wsc[:, None]).to(torch.float8_e4m3fn).view(torch.uint8)
        hq = th.float()
        hsc = hq.abs().amax(1).clamp_min(1e-30) / 448.0
        h8 = (hq / hsc[:, None]).to(torch.float8_e4m3fn).view(torch.uint8)
        return {"h": h8, "h_scale": hsc.contiguous()}, w8, {"w_scale": wsc.contiguous(),
                                                            "h_dtype": dg.DG_E4M3,
                                                            "w_dtype": dg.DG_E4M3}
    qw = dg.dg_quantize_nvfp4(tw)
    qh = dg.dg_quantize_nvfp4(th)
    return ({"h": qh["codes"], "h_scale": qh["scale"], "h_block_scale": qh["block_scale"]},
            qw["codes"], {"w_scale": qw["scale"], "w_block_scale": qw["block_scale"],
                          "h_dtype": dg.DG_NVFP4, "w_dtype": dg.DG_NVFP4, "d": d})


@pytest.mark.parametrize("precision,B,S,V,d", [
    ("bf16", 2, 100, 3001, 512),
    ("e4m3", 1, 256, 2000, 256),
    ("nvfp4", 1, 200, 1500, 512),
])
def test_host_step_matches_device_step(dg, precision, B, S, V, d):
    hd, w, kw = _case(dg, precision, B, S, V, d, 11 + V)
    torch.cuda.synchronize()
    R = B * S
    rng = np.random.default_rng(5)
    hh = {k: v.cpu().pin_memory() for k, v in hd.items()}
    w_scale = kw.pop("w_scale", None)
    dkw = dict(kw)
    desc = dg.host_desc(hh["h"], w, B=B, S=S, h_scale=hh.get("h_scale"),
                        h_block_scale=hh.get("h_block_scale"), w_scale=w_scale, **dkw)
    ws = torch.empty(dg.dg_workspace_bytes_host(desc), dtype=torch.uint8, device="cuda")
    K, seed, calls = 32, 9, 5
    canv = [torch.from_numpy(rng.integers(0, V, R).astype(np.int32)).pin_memory()
            for _ in range(calls)]
    outs = [torch.empty(R, dtype=torch.int32).pin_memory() for _ in range(calls)]
    means = [torch.empty(B, dtype=torch.float32).pin_memory() for _ in range(calls)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for i in range(calls):
        dg.dg_canvas_step_host(hh["h"], w, canv[i], K, seed, i, B=B, S=S, canvas_out=outs[i],
                               mean_entropy=means[i], workspace=ws, status=status, desc=desc)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    dev_kw = dict(kw)
    if "h_scale" in hd:
        dev_kw["h_scale"] = hd["h_scale"]
    if "h_block_scale" in hd:
        dev_kw["h_block_scale"] = hd["h_block_scale"]
    for i in range(calls):
        ref = dg.dg_canvas_step(hd["h"], w, canv[i].cuda(), K, seed, i, B=B, S=S,
                                w_scale=w_scale, **dev_kw)
        torch.cuda.synchronize()
        assert torch.equal(outs[i], ref["canvas"].cpu()), i
        assert torch.equal(means[i], ref["mean_entropy"].cpu()), i


def test_host_step_in_place_canvas(dg):
    """canvas_in and canvas_out may be the same host buffer: the upload precedes the read-back."""
    B, S, V, d = 1, 256, 4000, 256
    hd, w, _ = _case(dg, "bf16", B, S, V, d, 3)
    h = hd["h"].cpu().pin_memory()
    c0 = np.random.default_rng(1).integers(0, V, B * S).astype(np.int32)
    c = torch.from_numpy(c0.copy()).pin_memory()
    dg.dg_canvas_step_host(h, w, c, 32, 4, 0, B=B, S=S, canvas_out=c)
    torch.cuda.synchronize()
    ref = dg.dg_canvas_step(hd["h"], w, torch.from_numpy(c0).cuda(), 32, 4, 0, B=B, S=S)
    torch.cuda.synchronize()
    assert torch.equal(c, ref["canvas"].cpu())


def test_host_step_pageable_outputs(dg):
    """Outputs in pageable host memory and in page-locked host memory both receive the device
    step's results (the read-back copies are synchronous for the former)."""
    B, S, V, d = 2, 256, 3000, 256
    hd, w, _ = _case(dg, "bf16", B, S, V, d, 7)
    h = hd["h"].cpu().pin_memory()
    c0 = torch.from_numpy(np.random.default_rng(2).integers(0, V, B * S).astype(np.int32))
    out_pageable, mean_pageable = torch.empty(B * S, dtype=torch.int32), torch.empty(B)
    out_pinned = torch.empty(B * S, dtype=torch.int32).pin_memory()
    mean_pinned = torch.empty(B).pin_memory()
    dg.dg_canvas_step_host(h, w, c0.pin_memory(), 32, 4, 1, B=B, S=S, canvas_out=out_pageable,
                           mean_entropy=mean_pageable)
    dg.dg_canvas_step_host(h, w, c0.pin_memory(), 32, 4, 1, B=B, S=S, canvas_out=out_pinned,
                           mean_entropy=mean_pinned)
    torch.cuda.synchronize()
    ref = dg.dg_canvas_step(hd["h"], w, c0.cuda(), 32, 4, 1, B=B, S=S)
    torch.cuda.synchronize()
    for out, mean in ((out_pageable, mean_pageable), (out_pinned, mean_pinned)):
        assert torch.equal(out, ref["canvas"].cpu())
        assert torch.equal(mean, ref["mean_entropy"].cpu())
