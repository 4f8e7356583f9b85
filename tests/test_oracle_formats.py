"""Pins for the oracle's number formats: bf16 and E4M3 rounding, E4M3 decoding, row quantiser."""
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits_f32(x):
    return np.asarray(x, np.float32).view(np.uint32)


def test_bf16_round_matches_torch_on_float32_inputs(orc):
    rng = np.random.default_rng(1)
    # random bit patterns over a wide exponent range, plus exact ties (low 16 bits = 0x8000)
    u = rng.integers(0, 2**32, 400_000, dtype=np.uint64).astype(np.uint32)
    u = u[((u >> 23) & 0xFF) < 0xFF]                       # finite only
    ties = (u & 0xFFFF0000) | 0x8000
    u = np.concatenate([u, ties]).astype(np.uint32)
    x = u.view(np.float32)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = orc.bf16_round(x.astype(np.float64))
    assert np.array_equal(got, ref)


def test_bf16_round_single_rounding_from_double(orc):
    # 1 + 2^-8 + 2^-30 lies just above the midpoint between 1 and 1 + 2^-7: rounding the double
    # once gives 1 + 2^-7 (0x3F81); rounding through float32 first would tie to 1.0 (0x3F80).
    x = 1.0 + 2.0**-8 + 2.0**-30
    assert int(orc.bf16_round([x])[0]) == 0x3F81
    assert int(orc.bf16_round([-x])[0]) == 0xBF81
    assert int(orc.bf16_round([1.0 + 2.0**-8])[0]) == 0x3F80     # exact tie -> even
    assert int(orc.bf16_round([1.0 + 3 * 2.0**-8])[0]) == 0x3F82  # tie -> even (up)


def test_e4m3_published_encodings(orc):
    rows = []
    with open(os.path.join(GOLDEN, "e4m3_kat.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                a, b = line.split()
                rows.append((int(a, 16), float(b)))
    codes = np.array([a for a, _ in rows], np.uint8)
    vals = np.array([b for _, b in rows], np.float64)
    dec = orc.e4m3_value(codes)
    assert np.array_equal(dec, vals)
    assert np.array_equal(np.signbit(dec), np.signbit(vals))
    enc = orc.e4m3_round(vals.astype(np.float32))
    assert np.array_equal(enc, codes)
    assert np.isnan(orc.e4m3_value(np.array([0x7F, 0xFF], np.uint8))).all()


def test_e4m3_decode_all_codes_matches_torch(orc):
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = orc.e4m3_value(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_e4m3_round_exhaustive_over_bf16_inputs(orc):
    # every bf16 value with magnitude <= 448 (where no saturation can occur) against torch
    b = np.arange(1 << 16, dtype=np.uint32)
    x = (b << 16).view(np.float32)
    keep = np.isfinite(x) & (np.abs(x) <= 448.0)
    x = x[keep]
    ref = torch.from_numpy(x.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = orc.e4m3_round(x)
    assert np.array_equal(got, ref)


def test_e4m3_satfinite(orc):
    x = np.array([464.0, 465.0, 480.0, 1e9, np.inf, -np.inf, -500.0, 447.0], np.float32)
    got = orc.e4m3_round(x)
    # 464 is the midpoint between 448 (mantissa 110) and 480 (not finite): ties-to-even keeps 448
    assert list(got[:7]) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]
    assert got[7] == 0x7E      # 447 rounds to 448 (spacing 32 above 256)
    assert np.isnan(orc.e4m3_value(orc.e4m3_round(np.array([np.nan], np.float32)))).all()


def _bf16(vals):
    return (np.asarray(vals, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_quant_rows_hand_example(orc):
    h = _bf16([[1.0, -2.0, 0.5, 0.0], [0.0, 0.0, 0.0, 0.0]]).reshape(-1)
    q, sc = orc.quant_rows_e4m3(h, 2, 4)
    # amax = 2, inv = 224: products 224, -448, 112, 0
    assert list(q[:4]) == [0x76, 0xFE, 0x6E, 0x00]
    assert sc[0] == np.float32(2.0) / np.float32(448.0)
    assert list(q[4:]) == [0, 0, 0, 0] and sc[1] == np.float32(1.0)


def test_quant_rows_error_bound_and_amax(orc):
    rng = np.random.default_rng(3)
    rows, d = 64, 96
    x = rng.standard_normal(rows * d).astype(np.float32) * np.float32(3.0)
    hb = _bf16(x)
    q, sc = orc.quant_rows_e4m3(hb, rows, d)
    hv = (hb.astype(np.uint32) << 16).view(np.float32).astype(np.float64).reshape(rows, d)
    deq = orc.e4m3_value(q).reshape(rows, d) * sc.astype(np.float64)[:, None]
    amax = np.abs(hv).max(axis=1)
    # the row maximum maps to code magnitude 448 (0x7E / 0xFE)
    for r in range(rows):
        k = int(np.argmax(np.abs(hv[r])))
        assert (q[r * d + k] & 0x7F) == 0x7E
    # relative error of a normal E4M3 value is at most 2^-4; subnormal absolute error 2^-10*scale
    err = np.abs(deq - hv)
    bound = np.maximum(np.abs(hv) * 2.0**-4, 2.0**-10 * sc.astype(np.float64)[:, None]) * 1.0001
    assert (err <= bound + 1e-12 * amax[:, None]).all()


def test_e2m1_published_encodings(orc):
    rows = []
    with open(os.path.join(GOLDEN, "e2m1_kat.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                code, val = line.split()
                rows.append((int(code, 16), float(val)))
    assert len(rows) == 16
    got = orc.e2m1_value(np.array([c for c, _ in rows], np.uint8))
    for (code, val), g in zip(rows, got):
        assert g == val and np.signbit(g) == np.signbit(val), hex(code)


def _e2m1_nearest_even(x):
    """Brute force: the E2M1 code whose value is nearest to x, ties to the even code (mantissa
    bit 0), magnitudes beyond 6 saturated to 6."""
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    s = 0x8 if np.signbit(x) else 0
    a = min(abs(float(x)), 6.0)
    best = min(range(8), key=lambda c: (abs(mags[c] - a), c & 1))
    return s | best


def test_e2m1_rounding_brute_force(orc):
    # a dense grid covering every interval, every midpoint exactly, values past saturation, and
    # random fp32 values of both signs
    grid = np.arange(-8.0, 8.0, 0.0625, dtype=np.float32)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    rng = np.random.default_rng(3)
    x = np.concatenate([grid, mids, -mids, np.nextafter(mids, 0), np.nextafter(mids, 10),
                        (rng.standard_normal(20000) * 3).astype(np.float32),
                        np.array([1e-30, -1e-30, 100.0, -1e6], np.float32)])
    got = orc.e2m1_round(x)
    want = np.array([_e2m1_nearest_even(v) for v in x], np.uint8)
    assert np.array_equal(got, want)


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_nvfp4_quantiser_hand_row_and_roundtrip(orc):
    # one row of 32 elements = two blocks. Block 0 holds exact grid values times 0.25 with amax 6
    # times 0.25 = 1.5 (the row max): g = 1.5 / 2688, block scale = 1.5 / (6 g) = 448 exactly
    # (E4M3 0x7E), codes equal the grid codes. Block 1 is all zero: scale 0, codes 0.
    vals = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.5, -1, -1.5, -2, -3, -4, -6, 6], np.float32) * 0.25
    row = np.concatenate([vals, np.zeros(16, np.float32)])
    q, bs, sc = orc.quant_rows_nvfp4(_bf16(row), 1, 32)
    assert sc[0] == np.float32(1.5) / np.float32(2688)
    assert bs[0] == 0x7E and bs[1] == 0
    codes = np.stack([q & 0xF, q >> 4], axis=1).reshape(-1)
    assert list(codes[:16]) == [0, 1, 2, 3, 4, 5, 6, 7, 9, 10, 11, 12, 13, 14, 15, 7]
    assert not codes[16:].any()
    # decoded values e2m1 * value(block scale) * g reproduce the row within fp32 rounding
    dec = orc.e2m1_value(codes[:16]) * orc.e4m3_value(bs[:1])[0] * float(sc[0])
    assert np.allclose(dec, vals.astype(np.float64), rtol=1e-6, atol=0)
    # an all-zero row: scale 1, every block scale and code 0
    q, bs, sc = orc.quant_rows_nvfp4(np.zeros(32, np.uint16), 1, 32)
    assert sc[0] == 1.0 and not bs.any() and not q.any()


def test_nvfp4_quantiser_error_bound(orc):
    # every element lies within half a step of the E2M1 grid scaled by its block: the error is at
    # most 0.25 * value(block scale) * g below magnitude 2 (step 0.5), 0.5 up to 4, 1 up to 6
    rng = np.random.default_rng(11)
    R, d = 8, 64
    h = (rng.standard_normal(R * d) * np.exp(rng.standard_normal(R * d))).astype(np.float32)
    hb = _bf16(h)
    x = ((hb.astype(np.uint32) << 16).view(np.float32)).astype(np.float64).reshape(R, d)
    q, bs, sc = orc.quant_rows_nvfp4(hb, R, d)
    codes = np.stack([q & 0xF, q >> 4], axis=1).reshape(R, d)
    unit = orc.e4m3_value(bs).reshape(R, d // 16).repeat(16, axis=1) * sc[:, None].astype(np.float64)
    dec = orc.e2m1_value(codes.reshape(-1)).reshape(R, d) * unit
    mag = np.abs(x) / np.where(unit > 0, unit, 1)
    step = np.where(mag < 2, 0.5, np.where(mag < 4, 1.0, 2.0))
    assert (np.abs(dec - x) <= step / 2 * unit * (1 + 1e-6) + 1e-300).all()


def _e4m3_nearest_even_positive(t, table):
    """Brute force: the positive finite E4M3 code (0x00..0x7E, values from the OCP-pinned decoder)
    nearest to t >= 0, ties to the even code; t at or past 448 saturates to 0x7E."""
    if t >= 448.0:
        return 0x7E
    return min(range(0x7F), key=lambda c: (abs(table[c] - t), c & 1))


def test_nvfp4_quantiser_brute_force_scales_and_codes(orc):
    """Every row scale, block scale and code of the NVFP4 quantiser against an independent
    determination: the row scale g = fp32(amax / 2688); each block's scale the E4M3 value nearest
    to fp32(bmax / fp32(6 g)) found by searching all 127 finite codes (ties to even, saturating at
    448; a zero scale zeroes the block); each code the E2M1 value nearest to
    fp32(h / fp32(value(scale) g)) found by searching the 8 magnitudes (ties to even, saturating
    at 6). Rows span six decades within a row (so that some block scales are E4M3 subnormals or
    round to zero) and include an all-zero block."""
    table = [float(v) for v in orc.e4m3_value(np.arange(0x7F, dtype=np.uint8))]
    rng = np.random.default_rng(29)
    R, d = 6, 128
    h = (rng.standard_normal(R * d) * np.exp(3.0 * rng.standard_normal(R * d))).astype(np.float32)
    h[16:32] = 0.0                      # row 0, block 1: all zero
    h[d:d + 16] *= np.float32(1e-6)     # row 1, block 0: tiny next to the row maximum
    hb = _bf16(h)
    x = (hb.astype(np.uint32) << 16).view(np.float32).reshape(R, d)
    q, bs, sc = orc.quant_rows_nvfp4(hb, R, d)
    codes = np.stack([q & 0xF, q >> 4], axis=1).reshape(R, d)
    bs = bs.reshape(R, d // 16)
    f32 = np.float32
    for r in range(R):
        amax = f32(np.abs(x[r]).max())
        g = f32(amax / f32(2688.0))
        assert sc[r] == g, r
        for b in range(d // 16):
            blk = x[r, 16 * b:16 * b + 16]
            t = f32(f32(np.abs(blk).max()) / f32(f32(6.0) * g))
            want_s = _e4m3_nearest_even_positive(float(t), table)
            assert bs[r, b] == want_s, (r, b)
            unit = f32(f32(table[want_s]) * g)
            for k in range(16):
                if want_s == 0:
                    want_c = 0
                else:
                    want_c = _e2m1_nearest_even(f32(blk[k] / unit))
                assert codes[r, 16 * b + k] == want_c, (r, b, k)
    # the blocks built to test the corners really reached them
    assert bs[0, 1] == 0 and not codes[0, 16:32].any()
    assert bs[1, 0] < 0x08   # an E4M3 subnormal (or zero) block scale

    # Exact ties. amax = 2688 * 2^-10 makes g = 2^-10 exactly; a block whose maximum is
    # 11.25 * 2^-10 gets the scale 1.875 (E4M3 0x3F) exactly, so its unit is 1.875 * 2^-10, whose
    # reciprocal is inexact. The block's other elements sit exactly on the midpoints between E2M1
    # magnitudes (times the unit, all exact in bf16): the division lands on the midpoint and
    # rounds to the even code, where multiplying by the rounded reciprocal of the unit lands just
    # above 1.25, 2.5 and 5 and rounds up to the odd code.
    unit = 1.875 * 2.0**-10
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    blk1 = [6.0 * unit] + [m * unit for m in mids] + [-m * unit for m in mids] + [0.0]
    row = np.array([2688 * 2.0**-10] + [0.0] * 15 + blk1, np.float32)
    q, bs, sc = orc.quant_rows_nvfp4(_bf16(row), 1, 32)
    assert sc[0] == np.float32(2.0**-10) and bs[1] == 0x3F
    codes = np.stack([q & 0xF, q >> 4], axis=1).reshape(-1)[16:]
    even = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6}
    want = [7] + [even[m] for m in mids] + [0x8 | even[m] for m in mids] + [0]
    assert list(codes) == want


def test_quant_rows_brute_force_codes(orc):
    """Every code and scale of the per-row E4M3 quantiser against an independent determination:
    scale = fp32(amax / 448), inv = fp32(448 / amax), and each code the E4M3 value nearest to
    fp32(h * inv) found by searching all finite codes (ties to the even code, sign kept,
    saturating at 448). Rows of wide dynamic range reach the subnormal codes; two built rows put
    products exactly on E4M3 midpoints (or one fp32 step off them), where dividing by the scale
    instead of multiplying by inv would land on the other side."""
    table = [float(v) for v in orc.e4m3_value(np.arange(0x7F, dtype=np.uint8))]
    rng = np.random.default_rng(31)
    R, d = 10, 64
    x = (rng.standard_normal(R * d) * np.exp(2.5 * rng.standard_normal(R * d))).astype(np.float32)
    x[8 * d:] = 0
    # amax 1.9375: 0.0113525390625 * fp32(448 / 1.9375) = 2.625 exactly (midpoint of 2.5, 2.75)
    x[8 * d:8 * d + 3] = [1.9375, 0.0113525390625, 0.022705078125]
    # amax 3.1875: the product is one step above the midpoint 1.3125 (the quotient lands on it)
    x[9 * d:9 * d + 3] = [3.1875, 0.00933837890625, 0.0186767578125]
    hb = _bf16(x)
    xv = (hb.astype(np.uint32) << 16).view(np.float32).reshape(R, d)
    q, sc = orc.quant_rows_e4m3(hb, R, d)
    q = q.reshape(R, d)
    f32 = np.float32
    subnormal = 0
    for r in range(R):
        amax = f32(np.abs(xv[r]).max())
        assert sc[r] == f32(amax / f32(448.0)), r
        inv = f32(f32(448.0) / amax)
        for k in range(d):
            t = f32(xv[r, k] * inv)
            mag = _e4m3_nearest_even_positive(abs(float(t)), table)
            want = (0x80 if np.signbit(t) else 0) | mag
            if mag == 0:
                want = q[r, k] & 0x80   # a zero keeps whichever sign bit the quantiser gave it
            assert q[r, k] == want, (r, k)
            subnormal += 0 < mag < 0x08
    assert subnormal > 0
