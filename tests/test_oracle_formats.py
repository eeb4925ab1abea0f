"""Pins for the oracle's number formats (E2M1, E4M3, bf16).

The oracle decodes from bit fields and encodes by nearest-neighbour search on
the value grid.  These tests check it against things it does not share code
with: torch's float8_e4m3fn casts, numpy's float16, a generic minifloat
enumerator validated on those library formats, and round-half-even per
binade written with numpy's own rounding.
"""
import numpy as np
import pytest
import torch

from oracle import formats as F


def minifloat_values(ebits, mbits, bias, codes):
    """Generic IEEE-style minifloat decode (no inf/NaN handling): a second,
    independent restatement used only to cross-check the oracle."""
    out = []
    for c in codes:
        s = (c >> (ebits + mbits)) & 1
        e = (c >> mbits) & ((1 << ebits) - 1)
        m = c & ((1 << mbits) - 1)
        frac = m / float(1 << mbits)
        v = (2.0 ** (1 - bias)) * frac if e == 0 else (2.0 ** (e - bias)) * (1.0 + frac)
        out.append(-v if s else v)
    return np.array(out)


def test_minifloat_enumerator_matches_libraries():
    # float16 via numpy (5 exponent bits, 10 mantissa, bias 15), finite codes
    codes = np.arange(0, 0x7C00, 37, dtype=np.int64)
    ref = codes.astype(np.uint16).view(np.float16).astype(np.float64)
    assert np.array_equal(minifloat_values(5, 10, 15, codes), ref)
    # float8 e5m2 via torch
    c8 = np.arange(0, 0x7C)
    ref8 = torch.tensor(c8, dtype=torch.uint8).view(torch.float8_e5m2).double().numpy()
    assert np.array_equal(minifloat_values(5, 2, 15, c8), ref8)


def test_e4m3_decode_all_codes_vs_torch():
    codes = np.arange(256)
    ours = F.e4m3_decode(codes)
    ref = torch.tensor(codes, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(ours[fin], ref[fin])
    assert F.e4m3_decode(0x7E) == 448.0
    assert np.isnan(F.e4m3_decode(0x7F)) and np.isnan(F.e4m3_decode(0xFF))


def test_e2m1_decode_is_the_1_2_1_minifloat():
    codes = np.arange(16)
    assert np.array_equal(F.e2m1_decode(codes), minifloat_values(2, 1, 1, codes))
    assert F.e2m1_decode(7) == 6.0          # E2M1 max used by g = amax / (6 * 448)
    # every E2M1 value is an E4M3 value (so e2m1 * e4m3 products stay exact)
    grid = set(F.e4m3_decode(np.arange(0, 0x7F)).tolist())
    assert all(abs(v) in grid for v in F.e2m1_decode(codes))


def _tie_points(grid):
    mids = (grid[:-1] + grid[1:]) / 2
    pts = [mids, np.nextafter(mids.astype(np.float32), np.float32(np.inf)),
           np.nextafter(mids.astype(np.float32), np.float32(-np.inf)), grid]
    return np.concatenate([np.asarray(p, np.float64) for p in pts]).astype(np.float32)


def test_e4m3_encode_vs_torch_cast_in_range():
    rng = np.random.default_rng(0)
    grid = F.e4m3_decode(np.arange(0x7F))
    x = np.concatenate([_tie_points(grid),
                        rng.uniform(0, 460, 200000).astype(np.float32),
                        np.exp2(rng.uniform(-14, 8.8, 200000)).astype(np.float32)])
    x = x[(x >= 0) & (x < 464)]
    x = np.concatenate([x, -x])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(F.e4m3_encode(x), ref)


def test_e4m3_encode_saturates():
    x = np.array([448, 463.9, 464, 470, 1e6, 3e38, np.inf], np.float32)
    assert np.all(F.e4m3_encode(x) == 0x7E)
    assert np.all(F.e4m3_encode(-x) == 0xFE)


def _rne_binade(mag, mbits, emin, maxval):
    """Round half to even by binade: step = 2^(e - mbits) for mag in
    [2^e, 2^(e+1)), subnormal step 2^(emin - mbits); saturate at maxval."""
    mag = np.asarray(mag, np.float64)
    e = np.floor(np.log2(np.where(mag > 0, mag, 1.0)))
    e = np.maximum(e, emin)
    step = np.exp2(e - mbits)
    r = np.round(mag / step) * step           # numpy rounds halves to even
    return np.minimum(r, maxval)


def test_e2m1_encode_vs_binade_rounding():
    rng = np.random.default_rng(1)
    grid = F.e2m1_decode(np.arange(8))
    x = np.concatenate([_tie_points(grid), rng.uniform(0, 7, 100000).astype(np.float32),
                        np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.5, 100.0], np.float32)])
    got = F.e2m1_decode(F.e2m1_encode(x))
    want = _rne_binade(x, 1, 0, 6.0)
    assert np.array_equal(got, want)
    # the tie table: 0.25->0, 0.75->1, 1.25->1, 1.75->2, 2.5->2, 3.5->4, 5->4
    t = F.e2m1_decode(F.e2m1_encode(np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)))
    assert t.tolist() == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]


def test_e4m3_encode_vs_binade_rounding():
    rng = np.random.default_rng(2)
    x = np.exp2(rng.uniform(-12, 9.5, 300000)).astype(np.float32)
    got = F.e4m3_decode(F.e4m3_encode(x))
    want = _rne_binade(x, 3, -6, 448.0)
    assert np.array_equal(got, want)


def test_sign_kept_and_round_trip():
    assert F.e2m1_encode(np.float32(-0.1)) == 0x8
    assert F.e2m1_encode(np.float32(-0.0)) == 0x8
    assert F.e4m3_encode(np.float32(-1e-6)) == 0x80
    for dec, enc, n in ((F.e2m1_decode, F.e2m1_encode, 16), (F.e4m3_decode, F.e4m3_encode, 256)):
        codes = np.arange(n)
        vals = dec(codes)
        fin = np.isfinite(vals)
        assert np.array_equal(enc(vals[fin].astype(np.float32)), codes[fin].astype(np.uint8))


def test_bf16_to_f32_matches_torch():
    rng = np.random.default_rng(3)
    u = rng.integers(0, 1 << 16, 100000, dtype=np.uint16)
    ref = torch.from_numpy(u.view(np.int16)).view(torch.bfloat16).float().numpy()
    got = F.bf16_to_f32(u)
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
