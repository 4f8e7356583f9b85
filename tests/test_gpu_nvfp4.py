"""GPU parity of the NVFP4 (4-bit) head: the device quantiser and the scale packing against the
oracle and the documented layout, and the canvas pass on block-scaled E2M1 MMAs against the
oracle's exact contraction of the same NVFP4 values."""
import numpy as np
import pytest
import torch

from parity import TOL, check_select, check_stats, dev, dev_bf16, dev_u8, host

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


def _unpack_scales(packed, rows, d):
    """Invert the documented packed layout: chunk (G, s) at (G * d/256 + s) * 4096; row 256 G + m
    (l = m % 32, c = m / 32), block 16 s + 4 j + kb at byte
    (l / 8) * 1024 + j * 256 + (c / 4) * 128 + (l % 8) * 16 + (c % 4) * 4 + kb of the chunk."""
    nb, nsl = d // 16, d // 256
    r = np.arange(rows)[:, None]
    b = np.arange(nb)[None, :]
    G, m = r // 256, r % 256
    l, c = m % 32, m // 32
    s, j, kb = b // 16, (b // 4) % 4, b % 4
    off = ((G * nsl + s) * 4096 + (l // 8) * 1024 + j * 256 + (c // 4) * 128 + (l % 8) * 16 +
           (c % 4) * 4 + kb)
    return np.asarray(packed)[off]


def _codes(q):
    c = np.stack([q & 0xF, q >> 4], axis=-1).reshape(q.shape[0], -1)
    return np.where(c == 0x8, 0, c)      # -0 and +0 are the same value


def test_device_quantiser_matches_oracle(dg, orc):
    rng = np.random.default_rng(3)
    R, d = 300, 512
    x = (rng.standard_normal(R * d) * np.exp(2 * rng.standard_normal(R * d))).astype(np.float32)
    x[:d] = 0                         # an all-zero row
    x[d:d + 16] = 0                   # an all-zero block in a non-zero row
    x[2 * d:3 * d] *= 1e-30           # tiny values (subnormal block scales)
    # row 3: exact ties. g = 2^-10 (amax 2688 * 2^-10), a block of scale 1.875 (its maximum
    # 11.25 * 2^-10) whose elements sit on the midpoints between E2M1 magnitudes: the quotient by
    # the unit lands exactly on them and must round to the even code
    unit = 1.875 * 2.0**-10
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    x[3 * d:4 * d] = 0
    x[3 * d] = 2688 * 2.0**-10
    x[3 * d + 16:3 * d + 32] = [6.0 * unit] + [m * unit for m in mids] + [-m * unit for m in mids] + [0.0]
    hb = _bits(x)
    got = dg.dg_quantize_nvfp4(dev_bf16(hb, (R, d)))
    torch.cuda.synchronize()
    q, bs, sc = orc.quant_rows_nvfp4(hb, R, d)
    assert int(got["status"][0]) == 0
    assert np.array_equal(host(got["scale"]), sc)
    assert np.array_equal(_unpack_scales(host(got["block_scale"]), R, d), bs.reshape(R, d // 16))
    assert np.array_equal(_codes(host(got["codes"])), _codes(q.reshape(R, d // 2)))
    # rows past R in the padded scale array (R rounded up to 256) are zero
    padded = host(got["block_scale"])
    assert padded.size == dg.nvfp4_scale_bytes(R, d) == 512 * d // 16
    assert not _unpack_scales(padded, 512, d)[R:].any()


def test_pack_scales_layout(dg):
    rng = np.random.default_rng(4)
    rows, d = 300, 768
    plain = rng.integers(0, 255, rows * d // 16).astype(np.uint8)
    packed = host(dg.dg_nvfp4_pack_scales(dev_u8(plain, (rows, d // 16)), rows, d))
    torch.cuda.synchronize()
    assert packed.size == (rows + 255) // 256 * 256 * d // 16
    assert np.array_equal(_unpack_scales(packed, rows, d), plain.reshape(rows, d // 16))
    assert not _unpack_scales(packed, (rows + 255) // 256 * 256, d)[rows:].any()


def _nvfp4_case(dg, B, S, V, d, seed):
    from workloads import quantize_rows_nvfp4_bits
    rng = np.random.default_rng(seed)
    h = rng.standard_normal(B * S * d).astype(np.float32)
    w = (rng.standard_normal(V * d) / np.sqrt(d)).astype(np.float32)
    hb = _bits(h)
    wq, wbs, wsc = quantize_rows_nvfp4_bits(_bits(w), V, d)
    tw = dev_u8(wq, (V, d // 2))
    twb = dg.dg_nvfp4_pack_scales(dev_u8(wbs, (V, d // 16)), V, d)
    canvas = rng.integers(0, V, B * S).astype(np.int32)
    return hb, (wq, wbs, wsc), tw, twb, dev(wsc), canvas


@pytest.mark.parametrize("B,S,V,d", [
    (1, 256, 1000, 256),     # ragged vocabulary tail, one K slice
    (2, 100, 3001, 512),     # rows not a multiple of 128; canvases straddle row blocks
    (1, 64, 777, 768),       # short canvas
    (1, 256, 2083, 2816),    # full hidden size
    (3, 100, 1000, 256),     # 300 rows: three row blocks, the last holding 44 rows
    (1, 256, 600, 3328),     # 13 K slices, past the full hidden size
])
def test_nvfp4_pass_parity(dg, orc, B, S, V, d):
    hb, (wq, wbs, wsc), tw, twb, tws, canvas = _nvfp4_case(dg, B, S, V, d, V + d)
    K, seed, p = min(32, S), 5, 2
    res = dg.dg_canvas_step(dev_bf16(hb, (B * S, d)), tw, dev(canvas), K, seed, p, B=B, S=S,
                            w_scale=tws, w_dtype=dg.DG_NVFP4, w_block_scale=twb)
    torch.cuda.synchronize()
    g = {k: host(v) for k, v in res.items() if torch.is_tensor(v)}
    o = orc.step(B, S, V, d, "nvfp4", hb, wq, K, seed, p, w_scale=wsc, w_bscale=wbs)
    assert int(g["status"][0]) == 0
    check_stats(g, o, TOL["bf16"])
    check_select(g, o, B, S, V, K, seed, p, orc.draw)
    assert np.allclose(g["mean_entropy"], o["mean_entropy"], atol=TOL["bf16"])


@pytest.mark.parametrize("B,S", [(1, 256), (2, 100), (1, 64)])
def test_nvfp4_prequantised_h_matches_device_quantiser(dg, B, S):
    """NVFP4 h quantised by dg_quantize_nvfp4 and passed in directly (its packed block scales
    repacked into the head's row-block layout inside the pass) gives bit-identical statistics to
    bf16 h quantised inside the pass (straight into the row-block layout), including row counts
    that end inside a 128-row block."""
    V, d = 1500, 512
    hb, _, tw, twb, tws, canvas = _nvfp4_case(dg, B, S, V, d, 77)
    th = dev_bf16(hb, (B * S, d))
    a = dg.dg_canvas_stats(th, tw, B=B, S=S, w_scale=tws, w_dtype=dg.DG_NVFP4, w_block_scale=twb)
    qh = dg.dg_quantize_nvfp4(th)
    b = dg.dg_canvas_stats(qh["codes"], tw, B=B, S=S, w_scale=tws, h_scale=qh["scale"],
                           h_dtype=dg.DG_NVFP4, w_dtype=dg.DG_NVFP4, h_block_scale=qh["block_scale"],
                           w_block_scale=twb, d=d)
    torch.cuda.synchronize()
    for k in ("argmax", "conf", "entropy", "mean_entropy"):
        assert torch.equal(a[k], b[k]), k


def test_nvfp4_full_vocab_all_rows(dg, orc):
    """256 slots x 262144 vocab x d=2816 NVFP4 head in the launch configuration the benchmark
    times: every row against the oracle (on the same NVFP4 operands, h quantised by the oracle's
    rule), the kept set against the oracle's, the new canvas, the invariants."""
    from workloads import CONFIGS, make_pass_inputs
    cfg = CONFIGS["pass_nvfp4_v262144_d2816"]
    x = make_pass_inputs(cfg)
    tw = dev_u8(x["w"], (cfg.V, cfg.d // 2))
    twb = dg.dg_nvfp4_pack_scales(dev_u8(x["w_bscale"], (cfg.V, cfg.d // 16)), cfg.V, cfg.d)
    res = dg.dg_canvas_step(dev_bf16(x["h"], (cfg.R, cfg.d)), tw, dev(x["canvas"]), cfg.keep_k,
                            cfg.seed, 0, B=cfg.B, S=cfg.S, w_scale=dev(x["w_scale"]),
                            w_dtype=dg.DG_NVFP4, w_block_scale=twb)
    torch.cuda.synchronize()
    g = {k: host(v) for k, v in res.items() if torch.is_tensor(v)}
    o = orc.step(cfg.B, cfg.S, cfg.V, cfg.d, "nvfp4", x["h"], x["w"], cfg.keep_k, cfg.seed, 0,
                 w_scale=x["w_scale"], w_bscale=x["w_bscale"])
    check_stats(g, o, TOL["bf16"])
    check_select(g, o, cfg.B, cfg.S, cfg.V, cfg.keep_k, cfg.seed, 0, orc.draw)
    assert int(g["status"][0]) == 0
    assert (g["entropy"] >= 0).all() and (g["entropy"] <= np.log(cfg.V) + 1e-4).all()
    assert (g["conf"] >= 1.0 / cfg.V * 0.999).all() and (g["conf"] <= 1.0).all()
    assert abs(g["mean_entropy"][0] - o["mean_entropy"][0]) <= TOL["bf16"]
