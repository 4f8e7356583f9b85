"""Guard bands: every output, the workspace and the loop's hidden-state buffer are carved out of
larger device buffers whose margins hold a fill pattern; after a pass (or a whole loop) the
margins must be untouched, so no kernel writes outside the bytes it owns (the stand-in for a
memory checker, which is closed on this machine)."""
import numpy as np
import pytest
import torch

from parity import dev_bf16

pytestmark = pytest.mark.gpu

GUARD = 4096          # bytes of margin on each side (keeps 256-byte alignment of the interior)
FILL = 0xA5


@pytest.fixture(scope="module")
def dg():
    from uniform_state_denoising_vocab_b300 import build
    build.build()
    import uniform_state_denoising_vocab_b300 as m
    m.lib()
    return m


class Guarded:
    """A device byte buffer with GUARD margins; `view` is the interior as the requested dtype."""

    def __init__(self, nbytes, dtype, shape):
        inner = (nbytes + 255) // 256 * 256
        self.raw = torch.full((GUARD + inner + GUARD,), FILL, dtype=torch.uint8, device="cuda")
        self.nbytes = nbytes
        self.view = self.raw[GUARD:GUARD + nbytes].view(dtype).view(shape)

    def intact(self):
        r = self.raw.cpu().numpy()
        tail = r[GUARD + self.nbytes:]
        return bool((r[:GUARD] == FILL).all() and (tail == FILL).all())


def _g(n, dtype, shape=None):
    item = torch.empty(0, dtype=dtype).element_size()
    return Guarded(n * item, dtype, shape if shape is not None else (n,))


def _bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _step_guarded(dg, h, w, B, S, V, **kw):
    R = B * S
    rng = np.random.default_rng(3)
    canvas = torch.from_numpy(rng.integers(0, V, R).astype(np.int32)).cuda()
    outs = {"canvas": _g(R, torch.int32), "argmax": _g(R, torch.int32), "conf": _g(R, torch.float32),
            "entropy": _g(R, torch.float32), "kept": _g(R, torch.uint8),
            "mean_entropy": _g(B, torch.float32), "status": _g(1, torch.int32)}
    outs["status"].view.zero_()
    desc = dg.make_desc(h, w, B=B, S=S, **kw)
    ws = _g(dg.dg_workspace_bytes(desc), torch.uint8)
    import ctypes as C
    L = dg.lib()
    P = lambda t: C.c_void_p(t.data_ptr())
    rc = L.dg_canvas_step(C.byref(desc), P(canvas), P(outs["canvas"].view), 32, C.c_uint64(7),
                          C.c_uint32(1), P(outs["argmax"].view), P(outs["conf"].view),
                          P(outs["entropy"].view), P(outs["kept"].view),
                          P(outs["mean_entropy"].view), None, None, P(ws.view), ws.nbytes,
                          P(outs["status"].view), C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    assert int(outs["status"].view[0]) == 0
    for k, g in list(outs.items()) + [("workspace", ws)]:
        assert g.intact(), k


@pytest.mark.parametrize("B,S,V,d", [(1, 256, 3001, 256), (2, 100, 777, 512), (1, 64, 70000, 128)])
def test_step_bf16_writes_only_its_buffers(dg, B, S, V, d):
    rng = np.random.default_rng(V)
    h = dev_bf16(_bits(rng.standard_normal(B * S * d)), (B * S, d))
    w = dev_bf16(_bits(rng.standard_normal(V * d) / np.sqrt(d)), (V, d))
    _step_guarded(dg, h, w, B, S, V)


def test_step_e4m3_quantised_h_writes_only_its_buffers(dg):
    B, S, V, d = 2, 100, 2000, 256
    rng = np.random.default_rng(8)
    h = dev_bf16(_bits(rng.standard_normal(B * S * d)), (B * S, d))
    wf = torch.from_numpy((rng.standard_normal(V * d) / np.sqrt(d)).astype(np.float32)).view(V, d).cuda()
    wsc = (wf.abs().amax(1) / 448.0).contiguous()
    w8 = (wf / wsc[:, None]).to(torch.float8_e4m3fn).view(torch.uint8)
    _step_guarded(dg, h, w8, B, S, V, w_scale=wsc, w_dtype=dg.DG_E4M3)


def test_step_nvfp4_quantised_h_writes_only_its_buffers(dg):
    B, S, V, d = 2, 100, 1500, 512
    rng = np.random.default_rng(9)
    h = dev_bf16(_bits(rng.standard_normal(B * S * d)), (B * S, d))
    wq = dg.dg_quantize_nvfp4(dev_bf16(_bits(rng.standard_normal(V * d) / np.sqrt(d)), (V, d)))
    torch.cuda.synchronize()
    _step_guarded(dg, h, wq["codes"], B, S, V, w_scale=wq["scale"], w_dtype=dg.DG_NVFP4,
                  w_block_scale=wq["block_scale"])


def test_loop_writes_only_its_buffers(dg):
    """The whole loop (built-in denoiser, conditional graph): canvas, hidden-state buffer,
    statistics, state, status and workspace stay inside their bytes."""
    B, S, V, d = 2, 128, 4096, 256
    R = B * S
    rng = np.random.default_rng(11)
    w = dev_bf16(_bits(rng.standard_normal(V * d) / np.sqrt(d)), (V, d))
    y = torch.from_numpy(np.where(np.arange(R) % S < 50, rng.integers(1, V, R), 0).astype(np.int32)).cuda()
    canvas = _g(R, torch.int32)
    hbuf = _g(R * d, torch.bfloat16, (R, d))
    outs = {"argmax": _g(R, torch.int32), "conf": _g(R, torch.float32), "entropy": _g(R, torch.float32)}
    state = _g(B * 8, torch.int32, (B, 8))
    state.view.zero_()
    status = _g(1, torch.int32)
    status.view.zero_()
    desc = dg.make_desc(hbuf.view, w, B=B, S=S)
    ws = _g(dg.dg_workspace_bytes(desc), torch.uint8)
    res = dg.dg_canvas_loop(w, canvas.view, B=B, S=S, theta=0.05, y=y, h_buffer=hbuf.view,
                            state=state.view, status=status.view, workspace=ws.view,
                            outputs={k: g.view for k, g in outs.items()})
    torch.cuda.synchronize()
    assert int(status.view[0]) == 0
    assert int(dg.state_fields(res["state"])["passes"].min()) >= 1
    for k, g in [("canvas", canvas), ("h", hbuf), ("state", state), ("status", status),
                 ("workspace", ws)] + list(outs.items()):
        assert g.intact(), k
