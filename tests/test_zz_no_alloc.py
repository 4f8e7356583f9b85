"""dg_canvas_step_noalloc: the canvas pass for callers that cannot allocate device memory
(plugins whose host framework owns every device allocation, code that must not risk
cudaMalloc's implicit synchronisation or that runs under a fixed device-memory budget). Its
scratch is an array compiled into the library, so the caller passes only inputs and outputs.
Checked through the C ABI against the workspace-taking dg_canvas_step on two different calls in
a row (so a stale scratch from the first call would show in the second): both entry points run
the same kernels on the same inputs, so every output must be bit-identical. This file is
collected last on purpose."""
import ctypes as C

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dg():
    from uniform_state_denoising_vocab_b300 import build
    build.build()
    import uniform_state_denoising_vocab_b300 as m
    L = m.lib()
    vp = C.c_void_p
    L.dg_canvas_step_noalloc.argtypes = [C.POINTER(m.HeadDesc), vp, vp, C.c_int32, C.c_uint64,
                                         C.c_uint32, vp, vp, vp, vp, vp, vp,
                                         C.POINTER(m.StopRule), vp, vp]
    L.dg_canvas_step_noalloc.restype = C.c_int
    return m


def _case(B, S, V, d, seed):
    rng = np.random.default_rng(seed)
    h = torch.from_numpy(rng.standard_normal((B * S, d)).astype(np.float32)).to(torch.bfloat16).cuda()
    w = torch.from_numpy((rng.standard_normal((V, d)) / np.sqrt(d)).astype(np.float32)).to(torch.bfloat16).cuda()
    c = torch.from_numpy(rng.integers(0, V, B * S).astype(np.int32)).cuda()
    return h, w, c


def _noalloc(dg, h, w, canvas, B, S, K, seed, pass_, **desc_kw):
    R = B * S
    out = {"canvas": torch.empty(R, dtype=torch.int32, device="cuda"),
           "argmax": torch.empty(R, dtype=torch.int32, device="cuda"),
           "conf": torch.empty(R, device="cuda"), "entropy": torch.empty(R, device="cuda"),
           "kept": torch.empty(R, dtype=torch.uint8, device="cuda"),
           "mean_entropy": torch.empty(B, device="cuda"),
           "status": torch.zeros(1, dtype=torch.int32, device="cuda")}
    desc = dg.make_desc(h, w, B=B, S=S, **desc_kw)
    p = lambda t: C.c_void_p(t.data_ptr())
    rc = dg.lib().dg_canvas_step_noalloc(
        C.byref(desc), p(canvas), p(out["canvas"]), K, C.c_uint64(seed), C.c_uint32(pass_),
        p(out["argmax"]), p(out["conf"]), p(out["entropy"]), p(out["kept"]),
        p(out["mean_entropy"]), None, None, p(out["status"]),
        C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, dg.dg_status_string(rc)
    return out


def test_noalloc_matches_workspace_step_on_two_calls(dg):
    cases = [(1, 256, 3000, 256, 11, 0), (2, 200, 1700, 512, 12, 5)]
    inputs = [_case(B, S, V, d, seed) for (B, S, V, d, seed, _) in cases]
    # two calls in a row through the allocation-free entry point, on one stream
    got = [_noalloc(dg, h, w, c, B, S, 32, seed, p)
           for (h, w, c), (B, S, V, d, seed, p) in zip(inputs, cases)]
    # the same passes through the workspace-taking entry point
    ref = [dg.dg_canvas_step(h, w, c, 32, seed, p, B=B, S=S)
           for (h, w, c), (B, S, V, d, seed, p) in zip(inputs, cases)]
    torch.cuda.synchronize()
    for g, r in zip(got, ref):
        assert int(g["status"][0]) == 0
        for k in ("canvas", "argmax", "kept", "conf", "entropy", "mean_entropy"):
            assert torch.equal(g[k], r[k]), k


def test_noalloc_largest_workload_shape_that_fits(dg):
    """Eight 256-slot canvases (2048 rows, the batched workload's row count) with a vocabulary
    wide enough that the head splits it into as many groups as at V = 262144: the softmax
    partials take about 1.2 MB of the 4 MiB array (with 74 CTA pairs). Two calls in a row,
    bit-identical to dg_canvas_step."""
    B, S, V, d = 8, 256, 40000, 64
    h, w, c = _case(B, S, V, d, 13)
    desc = dg.make_desc(h, w, B=B, S=S)
    need = dg.dg_workspace_bytes(desc)
    assert need <= (4 << 20), need
    for seed, p in ((2, 0), (3, 1)):
        g = _noalloc(dg, h, w, c, B, S, 32, seed, p)
        r = dg.dg_canvas_step(h, w, c, 32, seed, p, B=B, S=S)
        torch.cuda.synchronize()
        assert int(g["status"][0]) == 0
        for k in ("canvas", "argmax", "kept", "conf", "entropy", "mean_entropy"):
            assert torch.equal(g[k], r[k]), k


@pytest.mark.parametrize("precision", ["e4m3", "nvfp4"])
def test_noalloc_quantised_heads_match_workspace_step(dg, precision):
    """bf16 hidden states against an E4M3 or NVFP4 head: the pass quantises h inside the array
    (quantised rows, row scales and, for NVFP4, the block scales in the head's layout) before the
    head reads it; two calls in a row, bit-identical to dg_canvas_step."""
    from workloads import quantize_rows_e4m3_bits, quantize_rows_nvfp4_bits
    B, S, V, d = 1, 256, 3000, 512
    rng = np.random.default_rng(21)
    h = torch.from_numpy(rng.standard_normal((B * S, d)).astype(np.float32)).to(torch.bfloat16).cuda()
    wf = torch.from_numpy((rng.standard_normal((V, d)) / np.sqrt(d)).astype(np.float32))
    wbits = wf.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).reshape(-1)
    c = torch.from_numpy(rng.integers(0, V, B * S).astype(np.int32)).cuda()
    if precision == "e4m3":
        wq, wsc = quantize_rows_e4m3_bits(wbits, V, d)
        w = torch.from_numpy(wq.reshape(V, d)).cuda()
        kw = {"w_scale": torch.from_numpy(wsc).cuda(), "w_dtype": dg.DG_E4M3}
    else:
        wq, wbs, wsc = quantize_rows_nvfp4_bits(wbits, V, d)
        w = torch.from_numpy(wq.reshape(V, d // 2)).cuda()
        twb = dg.dg_nvfp4_pack_scales(torch.from_numpy(wbs.reshape(V, d // 16)).cuda(), V, d)
        kw = {"w_scale": torch.from_numpy(wsc).cuda(), "w_dtype": dg.DG_NVFP4,
              "w_block_scale": twb}
    for seed, p in ((4, 0), (5, 1)):
        g = _noalloc(dg, h, w, c, B, S, 32, seed, p, **kw)
        r = dg.dg_canvas_step(h, w, c, 32, seed, p, B=B, S=S, **kw)
        torch.cuda.synchronize()
        assert int(g["status"][0]) == 0 and int(r["status"][0]) == 0
        for k in ("canvas", "argmax", "kept", "conf", "entropy", "mean_entropy"):
            assert torch.equal(g[k], r[k]), k


def test_noalloc_rejects_descriptors_beyond_its_scratch(dg):
    # an E4M3 head fed bf16 hidden states needs R*d bytes of quantised rows: far beyond the array
    V, d = 512, 2816
    w = torch.zeros(V, d, dtype=torch.uint8, device="cuda")
    ws = torch.ones(V, device="cuda")
    h = torch.zeros(16, d, dtype=torch.bfloat16, device="cuda")
    desc = dg.make_desc(h, w, B=64, S=1024, w_scale=ws)
    n = C.c_size_t(0)
    assert dg.lib().dg_workspace_bytes(C.byref(desc), C.byref(n)) == 0
    assert n.value > (4 << 20)
    c = torch.zeros(16, dtype=torch.int32, device="cuda")
    rc = dg.lib().dg_canvas_step_noalloc(C.byref(desc), C.c_void_p(c.data_ptr()),
                                         C.c_void_p(c.data_ptr()), 1, 0, 0, None, None, None, None,
                                         None, None, None, None, None)
    assert rc == -4   # DG_ERR_WORKSPACE, nothing enqueued
