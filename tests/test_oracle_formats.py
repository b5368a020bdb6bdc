"""Pins of the oracle's number formats and group quantisers (C1, C3).

Each check compares the oracle with something other than itself: the OCP
anchor values in tests/golden, torch's own fp32->float8_e4m3fn / bfloat16
conversions (a library routine), closed forms and hand-picked groups.
"""
import math
import os

import numpy as np
import pytest
import torch

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line.split()


def test_e2m1_decode_all_codes(orc):
    # OCP MX E2M1 grid, magnitude by 3-bit code, sign in bit 3
    grid = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for c in range(16):
        v = orc.e2m1_decode(c)
        assert abs(v) == grid[c & 7]
        assert math.copysign(1.0, v) == (-1.0 if c & 8 else 1.0)


def test_e2m1_encode_rne_golden(orc):
    for x, want in _rows("e2m1_rne.txt"):
        got = orc.e2m1_decode(orc.e2m1_encode(float(x)))
        assert got == float(want), (x, got, want)


def test_e2m1_roundtrip_and_negative_zero(orc):
    for c in range(16):
        assert orc.e2m1_encode(orc.e2m1_decode(c)) == c
    assert orc.e2m1_encode(-0.1) == 0x8  # rounds to zero, keeps the sign bit
    assert orc.e2m1_encode(0.1) == 0x0


def test_e4m3_decode_golden(orc):
    for code, want in _rows("e4m3_known.txt"):
        v = orc.e4m3_decode(int(code, 16))
        assert v == float(want) and math.copysign(1, v) == math.copysign(1, float(want))
    assert math.isnan(orc.e4m3_decode(0x7F)) and math.isnan(orc.e4m3_decode(0xFF))


def test_e4m3_decode_matches_torch_all_codes(orc):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        v = orc.e4m3_decode(c)
        if math.isnan(ref[c]):
            assert math.isnan(v)
        else:
            assert v == ref[c], c


def test_e4m3_encode_matches_torch(orc):
    rng = np.random.default_rng(7)
    xs = np.concatenate([
        rng.standard_normal(3000).astype(np.float32) * 20,
        rng.uniform(-448, 448, 2000).astype(np.float32),
        rng.uniform(-2 ** -6, 2 ** -6, 1000).astype(np.float32),  # subnormal range
        np.array([0.0, -0.0, 2 ** -10, 3 * 2 ** -11, 448.0, 447.9, 0.0146484375], np.float32),
    ])
    # all exact midpoints between neighbouring finite codes
    vals = torch.arange(127, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mids = ((vals[1:] + vals[:-1]) / 2).astype(np.float32)
    xs = np.concatenate([xs, mids, -mids])
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for x, r in zip(xs, ref):
        assert orc.e4m3_encode(float(x)) == int(r), (x, r)


def test_e4m3_satfinite(orc):
    assert orc.e4m3_encode(1e6) == 0x7E
    assert orc.e4m3_encode(-1e6) == 0xFE
    assert orc.e4m3_encode(460.0) == 0x7E


def test_e4m3_roundtrip_all_finite(orc):
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert orc.e4m3_encode(orc.e4m3_decode(c)) == c


def test_e8m0(orc):
    assert orc.e8m0_decode(127) == 1.0
    assert orc.e8m0_decode(128) == 2.0
    assert orc.e8m0_decode(0) == 2.0 ** -127
    assert orc.e8m0_decode(254) == 2.0 ** 127
    assert math.isnan(orc.e8m0_decode(255))


def test_bf16_matches_torch(orc):
    rng = np.random.default_rng(3)
    xs = np.concatenate([rng.standard_normal(4000).astype(np.float32) * 10,
                         np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -0.0, 1e-40], np.float32)])
    tb = torch.from_numpy(xs).to(torch.bfloat16)
    ref = tb.view(torch.int16).numpy().astype(np.uint16)
    back = tb.float().numpy()
    for x, r, b in zip(xs, ref, back):
        assert orc.bf16_encode(float(x)) == int(r)
        assert orc.bf16_decode(int(r)) == float(b)


# ---------------------------------------------------------------- groups (C3)
GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0, 6.0]


def test_nvfp4_identity_on_grid(orc):
    codes, sc = orc.nvfp4_quant16(GRID)
    assert orc.e4m3_decode(sc) == 1.0  # amax 6 -> scale exactly 1
    back = orc.dequant_nvfp4(codes[None], np.array([[sc]]))[0]
    assert list(back) == GRID


def test_nvfp4_max_2688(orc):
    # P4: with a per-16 E4M3 scale the largest representable value is 448 * 6
    x = np.array(GRID, np.float32) * 448
    codes, sc = orc.nvfp4_quant16(x)
    assert orc.e4m3_decode(sc) == 448.0
    back = orc.dequant_nvfp4(codes[None], np.array([[sc]]))[0]
    assert back.max() == 2688.0
    assert list(back) == list(x.astype(np.float64))


def test_nvfp4_post_rope_bound_does_not_saturate_scale(orc):
    # P4: post-RoPE KV stays within ~22.6, far below the 2688 range: the scale never saturates
    x = np.linspace(-22.6, 22.6, 16).astype(np.float32)
    codes, sc = orc.nvfp4_quant16(x)
    assert orc.e4m3_decode(sc) < 448
    back = orc.dequant_nvfp4(codes[None], np.array([[sc]]))[0]
    assert np.max(np.abs(back - x)) <= 0.5 * orc.e4m3_decode(sc) * 2 + 1e-6


def test_nvfp4_midpoints_even(orc):
    # unit scale (amax 6), midpoints between grid points go to the even code
    x = np.array([6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -1.25, -1.75, -2.5,
                  -3.5, -5.0, 0.0], np.float32)
    codes, sc = orc.nvfp4_quant16(x)
    back = orc.dequant_nvfp4(codes[None], np.array([[sc]]))[0]
    assert list(back) == [6.0, 0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, -0.0, -1.0, -1.0, -2.0, -2.0,
                          -4.0, -4.0, 0.0]


def test_nvfp4_zero_and_tiny_group(orc):
    codes, sc = orc.nvfp4_quant16(np.zeros(16))
    assert sc == 0 and not codes.any()
    # amax/6 below half the smallest E4M3 subnormal -> scale 0 -> all codes 0
    codes, sc = orc.nvfp4_quant16(np.full(16, 1e-3, np.float32))
    assert sc == 0 and not codes.any()


def test_nvfp4_error_bound_random(orc):
    # every value is within half a grid step (times the decoded scale) of its code,
    # unless it saturated at 6 * s
    rng = np.random.default_rng(11)
    for _ in range(200):
        x = rng.standard_normal(16).astype(np.float32) * rng.uniform(0.01, 50)
        codes, sc = orc.nvfp4_quant16(x)
        s = orc.e4m3_decode(sc)
        back = orc.dequant_nvfp4(codes[None], np.array([[sc]]))[0]
        y = x.astype(np.float64) / s
        step = np.where(np.abs(y) < 2, 0.5, np.where(np.abs(y) < 4, 1.0, 2.0))
        sat = np.abs(y) > 6
        assert np.all(sat | (np.abs(back / s - y) <= step / 2 + 1e-9))


def test_mxfp4_identity_on_scaled_grids(orc):
    for k in (-5, -2, 0, 1, 3, 7):
        x = np.array(GRID + GRID, np.float32) * np.float32(2.0 ** k)
        codes, sc = orc.mxfp4_quant32(x)
        assert sc == 127 + k
        back = orc.dequant_mxfp4(codes[None], np.array([[sc]]))[0]
        assert list(back) == list(x.astype(np.float64))


def test_mxfp4_scale_rule(orc):
    # e = floor(log2 amax) - 2, exactly at powers of two and just below them
    for amax, e in ((4.0, 0), (3.9999998, -1), (1.0, -2), (0.75, -3), (1024.0, 8)):
        x = np.zeros(32, np.float32)
        x[5] = amax
        _, sc = orc.mxfp4_quant32(x)
        assert sc - 127 == e, (amax, sc)
    codes, sc = orc.mxfp4_quant32(np.zeros(32))
    assert sc == 0 and not codes.any()


def test_mxfp8_identity_and_scale(orc):
    vals = torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    x = np.concatenate([vals[-16:], -vals[-16:]]).astype(np.float32)  # amax 448 -> e = 0
    codes, sc = orc.mxfp8_quant32(x)
    assert sc == 127
    back = np.array([orc.e4m3_decode(c) for c in codes])
    assert list(back) == list(x.astype(np.float64))
    x2 = x * np.float32(2.0 ** -6)
    codes2, sc2 = orc.mxfp8_quant32(x2)
    assert sc2 == 121 and list(codes2) == list(codes)


def test_encode_swa_matches_torch_route(orc):
    """The window slot ([P1] "890 bytes/token": window KV kept in 8 bits; reading:
    MXFP8, one E8M0 exponent per 32 values, e = floor(log2 amax) - 8) rebuilt by an
    independent route: the row's RoPE dims rotated, each 32-value block scaled by
    2^-e and cast by torch's float8_e4m3fn (clamped to +-448, the satfinite rule),
    the exponent read with numpy's frexp; bf16 slots by torch's bfloat16 cast."""
    rng = np.random.default_rng(31)
    for trial in range(40):
        v = (rng.standard_normal(576) * 2.0 ** rng.integers(-12, 12)).astype(np.float32)
        if trial % 5 == 0:
            v[rng.integers(0, 576, 40)] = 0.0
        if trial == 3:
            v[64:96] = 0.0  # an all-zero block: scale code 0, zero codes
        pos = int(rng.integers(0, 200000))
        cs = orc.rope_cs(1e4, pos)
        rot = v.copy()
        rot[512:] = orc.rope_apply(v[512:], cs)
        codes, scales = orc.encode_swa(v, cs, 1)
        for b in range(18):
            blk = rot[32 * b:32 * b + 32].astype(np.float64)
            amax = np.max(np.abs(blk))
            if amax == 0.0:
                assert scales[b] == 0 and not codes[32 * b:32 * b + 32].any()
                continue
            e = int(np.frexp(amax)[1]) - 1 - 8
            e = max(-127, min(127, e))
            assert scales[b] == e + 127, (trial, b)
            scaled = np.clip(np.ldexp(blk, -e), -448.0, 448.0)
            ref = torch.from_numpy(scaled.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(codes[32 * b:32 * b + 32], ref), (trial, b)
        hb, _ = orc.encode_swa(v, cs, 0)
        ref_bf16 = torch.from_numpy(rot).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(hb.view(np.uint16), ref_bf16), trial


def test_encode_entry_v4_independent_route(orc):
    """The V4 entry ([P5] §2.3.4: FP8 except the RoPE dims, kept bf16) rebuilt by
    an independent route: the 512 latent dims in 32-value blocks scaled by 2^-e
    (e = floor(log2 amax) - 8 from numpy's frexp) and cast by torch's
    float8_e4m3fn (clamped to +-448), the rotated RoPE dims by torch's bfloat16,
    the indexer key as in the V4.1 record."""
    rng = np.random.default_rng(43)
    for trial in range(20):
        v = (rng.standard_normal(576) * 2.0 ** rng.integers(-10, 10)).astype(np.float32)
        ik = rng.standard_normal(128).astype(np.float32)
        if trial == 2:
            v[32:64] = 0.0
        cs = orc.rope_cs(1e4, int(rng.integers(0, 100000)))
        lc, ls, rc, _, ic, isc = orc.encode_entry_v4(v, ik, cs)
        for b in range(16):
            blk = v[32 * b:32 * b + 32].astype(np.float64)
            amax = np.max(np.abs(blk))
            if amax == 0.0:
                assert ls[b] == 0 and not lc[32 * b:32 * b + 32].any()
                continue
            e = max(-127, min(127, int(np.frexp(amax)[1]) - 1 - 8))
            assert ls[b] == e + 127
            ref = torch.from_numpy(np.clip(np.ldexp(blk, -e), -448, 448).astype(np.float32)).to(
                torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(lc[32 * b:32 * b + 32], ref), (trial, b)
        rot = orc.rope_apply(v[512:], cs)
        ref_r = torch.from_numpy(rot).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(rc.view(np.uint16), ref_r)
        v41 = orc.encode_entry(v, ik, cs)
        assert np.array_equal(ic, v41[4]) and np.array_equal(isc, v41[5])


def test_attention_over_one_v4_entry_returns_its_latent(orc):
    """Attention over a single V4 entry (no window, no sink): the output is that
    entry's latent exactly, whatever the query -- values on the E4M3 grid times a
    power of two survive the encoding unchanged."""
    grid = torch.arange(0, 120, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    rng = np.random.default_rng(44)
    lat = (rng.choice(grid, 512) * rng.choice([-1.0, 1.0], 512)).astype(np.float32)
    lat[::32] = 448.0  # each block's amax: the scale is exactly 1
    v = np.concatenate([lat * np.float32(2.0 ** -3), rng.standard_normal(64).astype(np.float32)])
    c = orc.Cache(4, entry_format=orc.ENTRY_FP8)
    c.swa_codes[:] = 0
    rec = orc.encode_entry_v4(v, np.ones(128, np.float32), orc.rope_cs(1e4, 0))
    for arr, val in zip((c.lat_codes, c.lat_scales, c.rope_codes, c.rope_scales, c.idx_codes, c.idx_scales), rec):
        arr[0] = val
    c.n_tokens = c.n_entries = 1
    q = (rng.standard_normal((4, 576)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    out, lse = orc.sparse_attn(c, q, np.array([0, -1], np.int32), 1, 0.05,
                               swa_codes=np.zeros((0, 576), np.uint8), swa_scales=np.zeros((0, 18), np.uint8))
    for h in range(4):
        assert np.array_equal(out[h], lat * np.float32(2.0 ** -3))
