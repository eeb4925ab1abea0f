"""Exhaustive sweeps of the write path's hardware conversions against the
oracle's encoders, byte for byte.

The write kernel takes its E4M3 and E2M1 (and FP8) rounding decisions with
the hardware cvt.rn.satfinite conversions on IEEE FP32 quotients; the oracle
takes them by comparing distances to grid neighbours.  These sweeps put
every possible input through both:

  * every finite bf16 bit pattern (65,280 of them), sorted by magnitude and
    cut into 16-element blocks at all 16 offsets, so every value is once the
    maximum of its block (it sets the E4M3 block scale) and 15 times under a
    larger maximum (its E2M1 code is taken against another value's scale):
    4,080 tokens of one head of dimension 256, for NVFP4 at four global
    scales (1; the data's calibrated amax / 2688; one so large that the
    block scales fall into E4M3's subnormals or to zero; one so small that
    they saturate at 448), INT4 per-token-head, and FP8 per tensor at the
    same four scales;
  * every non-NaN E4M3 code (254) through the FP8-input write, the same
    block arrangement, at two input scales that are not powers of two, into
    NVFP4, INT4 and FP8 pools.

"SGLang's 4-bit KV cache", "The 56% survives its own scale": E2M1 elements
under one E4M3 scale per 16; "KV cache in 4 bits", "What we changed": the
INT4 per-token-head encoding.
"""
import numpy as np
import pytest
import torch

import bit_paged_kv_kv4_gb300 as K
from kv4_testlib import assert_guard_intact, dev_bf16, guarded_pool
from oracle import formats as F
from oracle import pool as OP

pytestmark = pytest.mark.gpu

D, P = 256, 16


def block_sweep(values):
    """`values` (any order) sorted by magnitude, then laid out 16 times, the
    i-th time shifted by i, so each value ends a 16-element block once; rows
    of D values (zero padded).  Returns the flat array [n_rows * D]."""
    order = np.argsort(np.abs(values.astype(np.float64)), kind="stable")
    v = values[order]
    n = v.size
    out = []
    for o in range(16):
        out.append(np.roll(v, -o))         # the element at o + 16j + 15 ends block j
    flat = np.concatenate(out)
    pad = (-flat.size) % D
    return np.concatenate([flat, np.zeros(pad, values.dtype)])


def finite_bf16():
    u = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    return u[((u >> 7) & 0xFF) != 0xFF]        # exponent all ones: inf / NaN


def run_write(fmt, k, v, g):
    T = k.shape[0]
    pages = (T + P - 1) // P
    pool = guarded_pool(fmt, pages, P, 1, D, fill=0x3C)
    slots = np.arange(T, dtype=np.int64)
    K.kv4_write(dev_bf16(k), dev_bf16(v), torch.from_numpy(slots).cuda(), pool, torch.from_numpy(g).cuda())
    torch.cuda.synchronize()
    assert K.kv4_device_error() == 0
    assert_guard_intact(pool.guard, "pool")
    spec = OP.PoolSpec(fmt, pages, P, 1, D)
    with np.errstate(over="ignore"):          # quotients past FP32's range saturate, as in the kernel
        ref = OP.write(OP.new_pool(spec, 0x3C), spec, k, v, slots, g)
    got = pool.buffer.cpu().numpy()
    diff = np.nonzero(got != ref)[0]
    assert diff.size == 0, f"{fmt} g={g}: {diff.size} bytes differ, first at {diff[:8]}"


@pytest.fixture(scope="module")
def bf16_rows():
    vals = finite_bf16()
    assert vals.size == 65280
    flat = block_sweep(vals)
    k = flat.reshape(-1, 1, D)
    # V: the same values, blocks in the reverse order of rows
    v = k[::-1].copy()
    return k, v


def scales(k, what):
    amax = float(np.abs(F.bf16_to_f32(k)).max())
    if what == "one":
        return np.float32(1.0)
    if what == "calibrated":
        return np.float32(np.float32(amax) / np.float32(2688.0))
    if what == "subnormal":
        return np.float32(2.0 ** 100)           # block maxima / (6 g) mostly under 2^-6
    return np.float32(2.0 ** -100)              # ... mostly above 448: saturate


@pytest.mark.parametrize("what", ["one", "calibrated", "subnormal", "saturating"])
def test_nvfp4_every_finite_bf16(bf16_rows, what):
    k, v = bf16_rows
    g = np.array([scales(k, what), scales(v, what)], np.float32)
    run_write("nvfp4", k, v, g)


def test_int4_every_finite_bf16(bf16_rows):
    k, v = bf16_rows
    run_write("int4", k, v, np.array([1.0, 1.0], np.float32))


@pytest.mark.parametrize("s", [1.0, 7.5e35, 2.0 ** 100, 2.0 ** -100])
def test_fp8_every_finite_bf16(bf16_rows, s):
    k, v = bf16_rows
    run_write("fp8", k, v, np.array([s, s * 1.5], np.float32))


@pytest.mark.parametrize("fmt", ["nvfp4", "int4", "fp8"])
@pytest.mark.parametrize("s_in", [0.37, 1.37])
def test_fp8_input_every_e4m3_code(fmt, s_in):
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    assert codes.size == 254
    flat = block_sweep(codes)
    k = flat.reshape(-1, 1, D)
    v = k[::-1].copy()
    T = k.shape[0]
    pages = (T + P - 1) // P
    s = np.array([s_in, s_in * 1.7], np.float32)
    g = np.array([0.0131, 0.0217], np.float32) if fmt != "fp8" else np.array([0.011, 0.019], np.float32)
    pool = guarded_pool(fmt, pages, P, 1, D, fill=0x3C)
    slots = np.arange(T, dtype=np.int64)
    K.kv4_write_fp8(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), torch.from_numpy(s).cuda(),
                    torch.from_numpy(slots).cuda(), pool, torch.from_numpy(g).cuda())
    torch.cuda.synchronize()
    assert K.kv4_device_error() == 0
    assert_guard_intact(pool.guard, "pool")
    spec = OP.PoolSpec(fmt, pages, P, 1, D)
    with np.errstate(over="ignore"):
        ref = OP.write_fp8(OP.new_pool(spec, 0x3C), spec, k, v, s, slots, g)
    got = pool.buffer.cpu().numpy()
    diff = np.nonzero(got != ref)[0]
    assert diff.size == 0, f"{fmt} s_in={s_in}: {diff.size} bytes differ, first at {diff[:8]}"


@pytest.mark.parametrize("fmt", ["nvfp4", "int4", "fp8"])
def test_every_finite_bf16_through_the_streamed_write(bf16_rows, fmt):
    """The same sweep three times over (12,240 tokens, 97,920 units of K and
    of V): more units than one pass of the resident grid has threads, so the
    write streams them through its shared-memory stages instead of taking
    its one-unit-a-thread form (the smaller sweeps above)."""
    k, v = bf16_rows
    k3 = np.concatenate([k, v, k])
    v3 = np.concatenate([v, k, v])
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert k3.shape[0] // 2 * (D // 16) > sms * 3 // 2 * 256      # units beyond one pass of the grid
    g = {"nvfp4": np.array([scales(k3, "calibrated")] * 2, np.float32),
         "int4": np.array([1.0, 1.0], np.float32),
         "fp8": np.array([0.0173, 0.0291], np.float32)}[fmt]
    run_write(fmt, k3, v3, g)
