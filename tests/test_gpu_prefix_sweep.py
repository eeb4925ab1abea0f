"""kv4_dequant_prefix over every block scale, every code and the extremes of
the global and FP8 scales, against the oracle, byte for byte.

The kernel computes each block's distinct dequantised values once and picks
every element's byte from them; these cases check that against the oracle's
per-element computation (x_hat in FP32, then E4M3(x_hat / s_fp8) with RNE and
saturation) where it is most likely to differ: every non-NaN E4M3 block scale
(both signs) under random codes, global scales that push x_hat into FP32's
subnormals or near its maximum, a negative global scale, and FP8 scales whose
reciprocal is subnormal or beyond 1e30 (the division's fallback path).

"SGLang's 4-bit KV cache", Figure 2: the 4-bit prefix is turned into FP8 in a
reused buffer before the extend attention; "The 56% survives its own scale":
the NVFP4 encoding (E2M1 elements under one E4M3 scale per 16, FP32 global
scale); "KV cache in 4 bits", "What we changed": the INT4 per-token-head
encoding.
"""
import numpy as np
import pytest
import torch

import bit_paged_kv_kv4_gb300 as K
import oracle
from kv4_testlib import assert_guard_intact, guarded_empty, guarded_pool
from oracle import pool as OP

pytestmark = pytest.mark.gpu

D, P, HKV, PAGES = 256, 16, 2, 8
E4M3_NOT_NAN = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)

G_VALUES = [1.0, 1.0 / 2688.0, 2.0 ** 100, 2.0 ** -100, -0.75]
S8_VALUES = [1.0, 0.37, 2.0 ** -100, 2.0 ** 100, 1.5 * 2.0 ** 127, 6.0e-39]


def sweep_pool(fmt, seed):
    """Random code bytes (every nibble value in every block scale's company);
    NVFP4 scale regions cycle through every non-NaN E4M3 byte, INT4 scales
    are FP32 values of both signs from 2^-140 to 2^120."""
    rng = np.random.default_rng(seed)
    spec = OP.PoolSpec(fmt, PAGES, P, HKV, D)
    pool = rng.integers(0, 256, spec.pool_bytes, dtype=np.uint8)
    n = P * spec.scale_bytes
    at = 0
    for page in range(PAGES):
        for h in range(HKV):
            for which in ("ks", "vs"):
                off = int(spec.chunk_offset(page, h)) + spec.region(which)
                if fmt == "nvfp4":
                    pool[off:off + n] = np.roll(E4M3_NOT_NAN, -at)[np.arange(n) % E4M3_NOT_NAN.size]
                    at += 37
                else:
                    e = rng.uniform(-140, 120, P)
                    s = (np.exp2(e) * rng.choice([-1.0, 1.0], P) * rng.uniform(1, 2, P)).astype(np.float32)
                    pool[off:off + n] = s.view(np.uint8)
    return spec, pool


def run_case(fmt, g, s8, seed):
    spec, host = sweep_pool(fmt, seed)
    table = np.random.default_rng(seed + 1).permutation(PAGES).astype(np.int32).reshape(2, PAGES // 2)
    prefix = np.array([PAGES // 2 * P, PAGES // 2 * P - 3], np.int32)
    cu = np.concatenate([[0], np.cumsum(prefix)]).astype(np.int64)
    gs = np.array([g, g * 1.25], np.float32)
    fs = np.array([s8, s8 * 0.75], np.float32)
    with np.errstate(over="ignore", under="ignore", invalid="ignore"):
        wk, wv = oracle.attention.dequant_prefix(host, spec, gs, table, prefix, fs)
    pool = guarded_pool(fmt, PAGES, P, HKV, D)
    pool.buffer.copy_(torch.from_numpy(host))
    total = int(prefix.sum())
    gk, gk_guard = guarded_empty((total, HKV, D), 0xEE)
    gv, gv_guard = guarded_empty((total, HKV, D), 0xEE)
    K.kv4_dequant_prefix(pool, torch.from_numpy(gs).cuda(), torch.from_numpy(table).cuda(),
                         torch.from_numpy(prefix).cuda(), torch.from_numpy(cu).cuda(), int(prefix.max()),
                         torch.from_numpy(fs).cuda(), gk, gv)
    torch.cuda.synchronize()
    assert K.kv4_device_error() == 0
    for name, got, want in (("K", gk, wk), ("V", gv, wv)):
        got = got.cpu().numpy()
        bad = np.nonzero(got.reshape(-1) != want.reshape(-1))[0]
        assert bad.size == 0, (f"{fmt} g={g} s8={s8} {name}: {bad.size} bytes differ, first at {bad[:4]}: "
                               f"{got.reshape(-1)[bad[:4]]} vs {want.reshape(-1)[bad[:4]]}")
    assert_guard_intact(gk_guard, "K workspace")
    assert_guard_intact(gv_guard, "V workspace")
    assert_guard_intact(pool.guard, "pool")


@pytest.mark.parametrize("s8", S8_VALUES)
@pytest.mark.parametrize("g", G_VALUES)
def test_nvfp4_every_block_scale(g, s8):
    run_case("nvfp4", g, s8, seed=5)


@pytest.mark.parametrize("s8", S8_VALUES)
def test_int4_scales_across_the_range(s8):
    run_case("int4", 1.0, s8, seed=6)
