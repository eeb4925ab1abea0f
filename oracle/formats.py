"""Number formats of the NVFP4 KV cache, written from their bit definitions.

Test infrastructure only (see ``oracle/__init__.py``).

Source: "SGLang's 4-bit KV cache: the 56% is exact, the 1.78x is untested",
Figure 2 caption (packed E2M1 K and V, one E4M3 block scale per sixteen
elements, per-layer FP32 global scales) and the section "The 56% survives its
own scale" (4-bit E2M1 element, FP8 E4M3 block scale, FP32 tensor scale).

Conventions fixed here (the pages name the formats, not their encoders):

* E2M1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0; exponent 0
  is subnormal (0 or 0.5).  Magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}.
* E4M3 (the "fn" variant used for FP8 KV): sign bit 7, exponent bits 6..3
  (bias 7), mantissa bits 2..0; exponent 0 is subnormal (m/8 * 2^-6); the code
  S.1111.111 is NaN; there is no infinity; largest finite 448.
* Encoders round to nearest, ties to the even code, and saturate to the
  largest finite magnitude ("satfinite").  The sign of the input is kept,
  also when the magnitude rounds to zero.

Encoders work on float32 inputs (the quantiser's arithmetic is FP32) and
choose between the two neighbouring grid values by comparing distances in
float64, which is exact for float32 inputs and grid values.
"""
import numpy as np

E2M1_MAX = 6.0
E4M3_MAX = 448.0


def e2m1_decode(codes):
    """E2M1 code (uint8 0..15, low nibble) -> float64 value."""
    c = np.asarray(codes).astype(np.int64) & 0xF
    sign = (c >> 3) & 1
    exp = (c >> 1) & 3
    man = c & 1
    mag = np.where(exp == 0, man * 0.5, (1.0 + man / 2.0) * np.exp2(exp - 1.0))
    return np.where(sign == 1, -mag, mag)


def e4m3_decode(codes):
    """E4M3 code (uint8 0..255) -> float64 value (NaN for S.1111.111)."""
    c = np.asarray(codes).astype(np.int64) & 0xFF
    sign = (c >> 7) & 1
    exp = (c >> 3) & 0xF
    man = c & 7
    mag = np.where(exp == 0, (man / 8.0) * 2.0 ** -6,
                   (1.0 + man / 8.0) * np.exp2(exp - 7.0))
    mag = np.where((exp == 15) & (man == 7), np.nan, mag)
    return np.where(sign == 1, -mag, mag)


# Non-negative finite grids, indexed by code (codes are monotone in value).
_E2M1_GRID = e2m1_decode(np.arange(8))            # codes 0..7
_E4M3_GRID = e4m3_decode(np.arange(127))          # codes 0..126 (0x7E = 448)


def _rne_on_grid(mag, grid):
    """Index of the grid value nearest to ``mag`` (>= 0), ties to even index,
    saturating at the last grid entry."""
    mag = np.asarray(mag, dtype=np.float64)
    top = len(grid) - 1
    lo = np.clip(np.searchsorted(grid, mag, side="right") - 1, 0, top)
    hi = np.minimum(lo + 1, top)
    d_lo = mag - grid[lo]
    d_hi = grid[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (lo % 2 == 1))
    idx = np.where(pick_hi, hi, lo)
    return np.where(mag >= grid[top], top, idx)


def e2m1_encode(x):
    """float32 array -> E2M1 codes (uint8), RNE, satfinite, sign kept."""
    x = np.asarray(x, dtype=np.float32)
    idx = _rne_on_grid(np.abs(x.astype(np.float64)), _E2M1_GRID)
    return (idx | (np.signbit(x).astype(np.int64) << 3)).astype(np.uint8)


def e4m3_encode(x):
    """float32 array -> E4M3 codes (uint8), RNE, satfinite, sign kept."""
    x = np.asarray(x, dtype=np.float32)
    idx = _rne_on_grid(np.abs(x.astype(np.float64)), _E4M3_GRID)
    return (idx | (np.signbit(x).astype(np.int64) << 7)).astype(np.uint8)


def bf16_to_f32(u16):
    """bf16 bit patterns (uint16) -> float32 (exact: bf16 is the top half)."""
    u = np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32)
