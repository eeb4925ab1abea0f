"""NVFP4 block quantisation and the INT4 per-token-head encoding.

Test infrastructure only (see ``oracle/__init__.py``).

NVFP4 ("SGLang's 4-bit KV cache", Figure 2 caption and "The 56% survives its
own scale"): each run of 16 consecutive elements along the head dimension
shares one E4M3 block scale; one FP32 global scale per layer (one for K, one
for V) is the outer level.  Nine bytes per sixteen values.

The pages do not print the encoder.  The reading used here, step by step in
IEEE float32 with round-to-nearest-even:

1. x = float32(bf16 input)                                       (exact)
2. amax = max |x_i| over the 16-element block
3. sf = amax / (6 * g)             -- 6 * g is rounded first, then the quotient
4. S = E4M3(sf), RNE, saturating at 448
5. denom = float32(S) * g;  if S == 0 or denom == 0 all 16 codes are +0
6. code_i = E2M1(x_i / denom), RNE, saturating at 6, sign kept
7. element 2j -> low nibble of byte j, element 2j+1 -> high nibble

Decode: x_hat = e2m1(code) * e4m3(S) * g  (exact in float64).

INT4 per-token-head ("KV cache in 4 bits", section "What we changed"): every
value in 4 bits, scale factors per token and attention head, 264 bytes per
head and token at head dim 256.  Reading: one FP32 symmetric scale for the K
row and one for the V row (2 x 4 = 8 bytes), s = amax / 7 (float32),
code = clamp(rne(x / s), -8, 7) as a two's-complement nibble, same packing;
amax == 0 (or s == 0) gives s = 0 and all-zero codes.  Decode: code * s.
The split of the eight scale bytes into two FP32 scales is a reading that
fits the byte count but that nothing on the pages confirms: parity unpinned
beyond the byte count.

FP8 E4M3 per tensor, the format the 4-bit cache is compared against ("SGLang's
4-bit KV cache", "The 56% survives its own scale": one scale for the whole
tensor and one byte per value, so 16 bytes per 16 values).  Reading: one FP32 decode scale s per
layer for K and one for V; code = E4M3(float32(x) / s), RNE, saturating at
448, sign kept.  Decode: e4m3(code) * s.
"""
import numpy as np

from .formats import bf16_to_f32, e2m1_decode, e2m1_encode, e4m3_decode, e4m3_encode

NVFP4_BLOCK = 16


def _pack_nibbles(codes):
    """[..., D] nibbles (0..15) -> [..., D/2] bytes, element 2j in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8) & 0xF
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def _unpack_nibbles(packed):
    """[..., D/2] bytes -> [..., D] nibbles (inverse of ``_pack_nibbles``)."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def _values(x):
    """Encoder input as float32: uint16 arrays are bf16 bit patterns, float32
    arrays are taken as they are (the FP8-input write's decoded values)."""
    x = np.asarray(x)
    if x.dtype == np.float32:
        return x
    assert x.dtype == np.uint16, x.dtype
    return bf16_to_f32(x)


def fp8_input_values(codes, s_in):
    """The FP8-input write's values: e4m3(code) * s_in as one IEEE float32
    product (round to nearest), the engine's FP8 K/V with its per-tensor
    scale ("SGLang's 4-bit KV cache", Figure 2: the K/V handed to the cache
    are FP8)."""
    return (e4m3_decode(np.asarray(codes)).astype(np.float32) * np.float32(s_in)).astype(np.float32)


def nvfp4_quantize(x_bf16, g):
    """Quantise rows of bf16 bit patterns (or float32 values) to NVFP4.

    x_bf16: uint16 [..., D] (D a multiple of 16); g: float32 global scale > 0.
    Returns (codes uint8 [..., D/2], scales uint8 [..., D/16]).
    """
    x = _values(x_bf16)
    D = x.shape[-1]
    assert D % NVFP4_BLOCK == 0
    g = np.float32(g)
    blocks = x.reshape(x.shape[:-1] + (D // NVFP4_BLOCK, NVFP4_BLOCK))
    amax = np.max(np.abs(blocks), axis=-1)                      # float32
    sf = (amax / (np.float32(6.0) * g)).astype(np.float32)      # step 3
    S = e4m3_encode(sf)                                          # step 4
    denom = (e4m3_decode(S).astype(np.float32) * g).astype(np.float32)  # step 5
    zero_block = (S == 0) | (denom == 0)
    safe = np.where(zero_block, np.float32(1.0), denom).astype(np.float32)
    q = (blocks / safe[..., None]).astype(np.float32)           # step 6
    codes = e2m1_encode(q)
    codes = np.where(zero_block[..., None], np.uint8(0), codes)
    return _pack_nibbles(codes.reshape(x.shape)), S


def nvfp4_dequantize(codes, scales, g):
    """NVFP4 bytes -> float64 values [..., D]: e2m1 * e4m3 * g."""
    vals = e2m1_decode(_unpack_nibbles(codes))
    D = vals.shape[-1]
    s = e4m3_decode(scales).astype(np.float64)
    vals = vals.reshape(vals.shape[:-1] + (D // NVFP4_BLOCK, NVFP4_BLOCK)) * s[..., None]
    return vals.reshape(vals.shape[:-2] + (D,)) * np.float64(np.float32(g))


def int4_quantize(x_bf16):
    """INT4 per-token-head: rows of bf16 (or float32) -> (codes uint8 [..., D/2], scale f32 [...])."""
    x = _values(x_bf16)
    amax = np.max(np.abs(x), axis=-1)
    s = (amax / np.float32(7.0)).astype(np.float32)
    safe = np.where(s == 0, np.float32(1.0), s).astype(np.float32)
    q = np.rint((x / safe[..., None]).astype(np.float32))
    c = np.clip(q, -8, 7).astype(np.int64)
    c = np.where((s == 0)[..., None], 0, c)
    return _pack_nibbles((c & 0xF).astype(np.uint8)), s


def int4_dequantize(codes, scale):
    """INT4 bytes + per-row scale -> float64 values."""
    n = _unpack_nibbles(codes).astype(np.int64)
    c = np.where(n >= 8, n - 16, n)
    return c * np.asarray(scale, dtype=np.float64)[..., None]


def fp8_quantize(x_bf16, s):
    """bf16 bits [..., D] -> E4M3 codes uint8 [..., D]: E4M3(x / s), the FP32
    quotient rounded to nearest, then RNE onto the E4M3 grid with saturation."""
    x = _values(x_bf16)
    return e4m3_encode((x / np.float32(s)).astype(np.float32))


def fp8_dequantize(codes, s):
    """E4M3 codes -> float64 values e4m3(code) * s."""
    return e4m3_decode(codes) * np.float64(np.float32(s))


def calibrate_global_scale(x_bf16):
    """Serving-time calibration of one NVFP4 global scale ("SGLang's 4-bit KV
    cache": Figure 2 keeps per-layer FP32 global scales; the measured runs
    went without them, and calibrating them is named there as unfinished
    work).  Reading:
    the tensor's absolute maximum mapped onto E2M1 max x E4M3 max,
    g = float32(amax) / 2688 (one FP32 rounding), and g = 1 when amax is not
    positive (an all-zero tensor encodes to zeros whatever g is)."""
    x = bf16_to_f32(np.asarray(x_bf16))
    amax = np.float32(np.max(np.abs(x))) if x.size else np.float32(0.0)
    return np.float32(amax / np.float32(2688.0)) if amax > 0 else np.float32(1.0)
