"""kv4_write on the GPU against the oracle's encoder: packed codes and scales
must match byte for byte (NVFP4, INT4 and FP8), including crafted rounding ties,
zero blocks, saturating blocks and skipped / out-of-range slots."""
import numpy as np
import pytest
import torch

import bit_paged_kv_kv4_gb300 as K
from kv4_testlib import Case, assert_guard_intact, dev_bf16, guarded_pool
from oracle import formats as F
from oracle import pool as OP
from workloads import TINY, f32_to_bf16_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fmt", ["nvfp4", "int4", "fp8"])
@pytest.mark.parametrize("D,P", [(64, 16), (128, 32), (256, 64), (256, 1600)])
def test_write_bit_exact(fmt, D, P):
    c = Case(fmt, 2, 4, D, [37, 300, 1], P, seed=D + P, outlier_ch=(3, 77 % D))
    pool = c.gpu_pool(fill=0xA5)
    _, ref = c.oracle_pool(fill=0xA5)
    got = pool.buffer.cpu().numpy()
    assert K.kv4_device_error() == 0
    assert_guard_intact(pool.guard, "pool")
    diff = np.nonzero(got != ref)[0]
    assert diff.size == 0, f"{diff.size} bytes differ, first at {diff[:8]}"


def test_write_tiny_workload_exact():
    w = TINY
    L = int(w.seq_lens()[0])
    num_pages, table = w.block_table(w.seq_lens())
    k, v = w.kv_request(0, 0, L)
    k, v = k[:, None], v[:, None]
    from workloads import global_scale_from_amax, slots_for
    g = np.array([global_scale_from_amax(np.abs(F.bf16_to_f32(k)).max()),
                  global_scale_from_amax(np.abs(F.bf16_to_f32(v)).max())], np.float32)
    slots = slots_for(table[0], w.page_size, np.arange(L))
    spec = OP.PoolSpec("nvfp4", num_pages, w.page_size, 1, w.head_dim)
    ref = OP.new_pool(spec, 0)
    OP.write(ref, spec, k, v, slots, g)
    pool = K.Pool("nvfp4", num_pages, w.page_size, 1, w.head_dim)
    pool.buffer.zero_()
    K.kv4_write(dev_bf16(k), dev_bf16(v), torch.from_numpy(slots).cuda(), pool, torch.from_numpy(g).cuda())
    assert np.array_equal(pool.buffer.cpu().numpy(), ref)


def _tie_rows(D=256):
    """Rows whose blocks hit E4M3 and E2M1 rounding ties with g = 1."""
    rows = []
    # E4M3 ties: block amax = 6 * (midpoint of two E4M3 neighbours), exact in bf16
    grid = F.e4m3_decode(np.arange(0x7F))
    mids = (grid[:-1] + grid[1:]) / 2
    for m in mids:
        amax = np.float32(6.0 * m)
        if F.bf16_to_f32(f32_to_bf16_bits(np.array([amax], np.float32)))[0] != amax:
            continue
        rows.append(np.full(16, amax / 3, np.float32))
        rows[-1][0] = amax
    # E2M1 ties: scale exactly 1 (amax 6), elements on every tie and neighbour
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -5.0, 6.0, -6.0,
                     1e-30, -1e-30, 0.0, -0.0], np.float32)
    for sc in (1.0, 2.0 ** -6, 2.0 ** -9, 448.0 / 64):
        rows.append(ties * np.float32(sc))
    # all-zero block, tiny block (scale rounds to 0), huge block (saturating scale)
    rows.append(np.zeros(16, np.float32))
    rows.append(np.full(16, 1e-20, np.float32))
    rows.append(np.linspace(-3e4, 3e4, 16).astype(np.float32))
    blocks = np.stack(rows)
    n = (len(blocks) + D // 16 - 1) // (D // 16) * (D // 16)
    blocks = np.concatenate([blocks, np.zeros((n - len(blocks), 16), np.float32)])
    return blocks.reshape(-1, D)


@pytest.mark.parametrize("g", [1.0, 0.01, 3.0])
def test_write_rounding_ties_exact(g):
    x = f32_to_bf16_bits(_tie_rows())
    T = x.shape[0]
    k = x[:, None]
    v = x[::-1].copy()[:, None]
    spec = OP.PoolSpec("nvfp4", (T + 15) // 16, 16, 1, 256)
    slots = np.arange(T, dtype=np.int64)
    gs = np.array([g, g], np.float32)
    ref = OP.new_pool(spec, 0)
    OP.write(ref, spec, k, v, slots, gs)
    pool = K.Pool("nvfp4", spec.num_pages, 16, 1, 256)
    pool.buffer.zero_()
    K.kv4_write(dev_bf16(k), dev_bf16(v), torch.from_numpy(slots).cuda(), pool, torch.from_numpy(gs).cuda())
    got = pool.buffer.cpu().numpy()
    diff = np.nonzero(got != ref)[0]
    assert diff.size == 0, f"{diff.size} bytes differ, first at {diff[:8]}"


def test_write_skips_negative_and_flags_out_of_range_slots():
    c = Case("nvfp4", 1, 1, 64, [20], 16, seed=5)
    slots = c.slots.copy()
    slots[3] = -1
    slots[5] = c.num_pages * 16 + 7          # beyond the pool: skipped, flagged
    pool = guarded_pool("nvfp4", c.num_pages, 16, 1, 64, fill=0x5A)
    g = torch.from_numpy(c.g).cuda()
    K.kv4_device_error()
    K.kv4_write(dev_bf16(c.k), dev_bf16(c.v), torch.from_numpy(slots).cuda(), pool, g)
    assert K.kv4_device_error() == 4          # KV4_EBOUNDS
    assert K.kv4_device_error() == 0          # cleared by the read
    spec = OP.PoolSpec("nvfp4", c.num_pages, 16, 1, 64)
    ref = OP.new_pool(spec, 0x5A)
    keep = slots.copy()
    keep[5] = -1
    OP.write(ref, spec, c.k, c.v, keep, c.g)
    assert np.array_equal(pool.buffer.cpu().numpy(), ref)
    assert_guard_intact(pool.guard, "pool")             # the slot past the end went nowhere


@pytest.mark.parametrize("fmt", ["nvfp4", "int4", "fp8"])
@pytest.mark.parametrize("D", [64, 256])
def test_write_fp8_input_bit_exact(fmt, D):
    """kv4_write_fp8 (FP8 E4M3 K/V with per-tensor input scales, non-power-of-
    two so the products round) against the oracle's write_fp8, byte for byte."""
    from workloads import fp8_kv_codes
    T, H, P, pages = 300, 2, 16, 24
    codes, s_in = fp8_kv_codes(D, T, H, D, "cuda", [[1, 5]] * H, 9.0)
    s_in = (s_in * np.float32(1.37)).astype(np.float32)
    rng = np.random.default_rng(D)
    slots = rng.permutation(pages * P)[:T].astype(np.int64)
    slots[::17] = -1                                    # skipped tokens
    g = np.array([0.013, 0.021], np.float32)
    pool = guarded_pool(fmt, pages, P, H, D, fill=0x5A)
    K.kv4_write_fp8(codes[0].contiguous(), codes[1].contiguous(), torch.from_numpy(s_in).cuda(),
                    torch.from_numpy(slots).cuda(), pool, torch.from_numpy(g).cuda())
    torch.cuda.synchronize()
    assert K.kv4_device_error() == 0
    spec = OP.PoolSpec(fmt, pages, P, H, D)
    ref = OP.write_fp8(OP.new_pool(spec, 0x5A), spec, codes[0].cpu().numpy(), codes[1].cpu().numpy(),
                       s_in, slots, g)
    got = pool.buffer.cpu().numpy()
    diff = np.nonzero(got != ref)[0]
    assert diff.size == 0, f"{diff.size} bytes differ, first at {diff[:8]}"
    assert_guard_intact(pool.guard, "pool")


@pytest.mark.parametrize("fmt", ["nvfp4", "int4"])
@pytest.mark.parametrize("D", [64, 256])
def test_write_pair_rows_every_slot_pattern(fmt, D):
    """A thread writes tokens 2p and 2p+1 of the call; NVFP4 and INT4 V
    store both halves of a pair row at once only when they land in one, and
    otherwise write each token's own part (NVFP4: its nibbles, set
    atomically; INT4: its 16-bit halves), keeping its partner's.
    One call mixes: an aligned run (plain stores), a run starting at an odd
    offset, pair rows whose halves come from non-adjacent tokens, a reversed
    pair, a skipped token beside a written partner, and an odd token count
    (the last token alone) -- over a pool of random bytes, whose untouched
    nibbles and rows must survive."""
    P, H = 16, 2
    slots = np.array([32, 33, 34, 35, 36, 37,      # aligned: pair rows 16..18
                      5, 6, 7, 8,                  # odd start: halves of rows 2..4
                      10, 13, 11, 12,              # rows 5 and 6 from non-adjacent tokens
                      21, 20,                      # reversed pair
                      44, -1,                      # a written even half, a skipped partner
                      50, 51, 52], np.int64)       # odd count: 52 is alone
    T = slots.size
    rng = np.random.default_rng(D)
    x = (rng.standard_normal((2, T, H, D)) * np.exp(rng.uniform(-3, 3, (2, T, H, 1)))).astype(np.float32)
    x[:, :, :, 5] *= 9.0
    k, v = f32_to_bf16_bits(x[0]), f32_to_bf16_bits(x[1])
    g = np.array([np.abs(x[0]).max() / 2688.0, np.abs(x[1]).max() / 2688.0], np.float32)
    pages = 4
    spec = OP.PoolSpec(fmt, pages, P, H, D)
    fill = rng.integers(0, 256, spec.pool_bytes, dtype=np.uint8)
    if fmt == "int4":
        # keep the untouched scale words finite
        for page in range(pages):
            for h in range(H):
                off = int(spec.chunk_offset(page, h)) + spec.region("ks")
                fill[off:off + 2 * P * 4] = np.full(2 * P, 0.5, np.float32).view(np.uint8)
    ref = OP.write(fill.copy(), spec, k, v, slots, g)
    pool = guarded_pool(fmt, pages, P, H, D)
    pool.buffer.copy_(torch.from_numpy(fill))
    K.kv4_write(dev_bf16(k), dev_bf16(v), torch.from_numpy(slots).cuda(), pool, torch.from_numpy(g).cuda())
    torch.cuda.synchronize()
    assert K.kv4_device_error() == 0
    assert_guard_intact(pool.guard, "pool")
    got = pool.buffer.cpu().numpy()
    diff = np.nonzero(got != ref)[0]
    assert diff.size == 0, f"{fmt} D{D}: {diff.size} bytes differ, first at {diff[:8]}"


@pytest.mark.parametrize("fmt", ["nvfp4", "int4", "fp8"])
@pytest.mark.parametrize("D", [64, 128, 256])
def test_write_many_units_per_thread(fmt, D):
    """A prefill-sized call: each thread of the resident grid walks several
    units through its staging ring (12,289 tokens x 4 heads x D/16 blocks per
    K|V: up to about seven units a thread at D = 256, and more units than one
    pass of the grid at every D).  An aligned run, a shuffled run with skipped
    tokens and the odd last token, over a pool of random bytes."""
    T, H, P = 12289, 4, 64
    pages = (T + P - 1) // P + 8
    rng = np.random.default_rng(12289)
    x = (rng.standard_normal((2, T, H, D)) * np.exp(rng.uniform(-3, 3, (2, T, H, 1)))).astype(np.float32)
    x[:, :, :, 9] *= 11.0
    k, v = f32_to_bf16_bits(x[0]), f32_to_bf16_bits(x[1])
    g = np.array([np.abs(x[0]).max() / 2688.0, np.abs(x[1]).max() / 2688.0], np.float32)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert (T + 1) // 2 * H * (D // 16) > sms * 3 // 2 * 256      # the streamed form
    half = 6000
    slots = np.concatenate([np.arange(half) + 2 * P,
                            rng.permutation(np.arange(half + 2 * P + 1, pages * P))[:T - half]]).astype(np.int64)
    slots[half::13] = -1
    spec = OP.PoolSpec(fmt, pages, P, H, D)
    fill = rng.integers(0, 256, spec.pool_bytes, dtype=np.uint8)
    if fmt == "int4":
        for page in range(pages):
            for h in range(H):
                off = int(spec.chunk_offset(page, h)) + spec.region("ks")
                fill[off:off + 2 * P * 4] = np.full(2 * P, 0.5, np.float32).view(np.uint8)
    ref = OP.write(fill.copy(), spec, k, v, slots, g)
    pool = guarded_pool(fmt, pages, P, H, D)
    pool.buffer.copy_(torch.from_numpy(fill))
    K.kv4_write(dev_bf16(k), dev_bf16(v), torch.from_numpy(slots).cuda(), pool, torch.from_numpy(g).cuda())
    torch.cuda.synchronize()
    assert K.kv4_device_error() == 0
    assert_guard_intact(pool.guard, "pool")
    got = pool.buffer.cpu().numpy()
    diff = np.nonzero(got != ref)[0]
    assert diff.size == 0, f"{fmt}: {diff.size} bytes differ, first at {diff[:8]}"


def test_write_fp8_input_many_units_per_thread():
    """The FP8-input write (16 staged bytes a token) at prefill size: several
    units per thread through the staging ring, byte for byte."""
    from workloads import fp8_kv_codes
    T, H, D, P = 12289, 4, 256, 64
    pages = (T + P - 1) // P + 4
    codes, s_in = fp8_kv_codes(77, T, H, D, "cuda", [[2, 40]] * H, 12.0)
    s_in = (s_in * np.float32(0.73)).astype(np.float32)
    rng = np.random.default_rng(77)
    slots = rng.permutation(pages * P)[:T].astype(np.int64)
    slots[::29] = -1
    g = np.array([0.017, 0.009], np.float32)
    pool = guarded_pool("nvfp4", pages, P, H, D, fill=0x3C)
    K.kv4_write_fp8(codes[0].contiguous(), codes[1].contiguous(), torch.from_numpy(s_in).cuda(),
                    torch.from_numpy(slots).cuda(), pool, torch.from_numpy(g).cuda())
    torch.cuda.synchronize()
    assert K.kv4_device_error() == 0
    spec = OP.PoolSpec("nvfp4", pages, P, H, D)
    ref = OP.write_fp8(OP.new_pool(spec, 0x3C), spec, codes[0].cpu().numpy(), codes[1].cpu().numpy(),
                       s_in, slots, g)
    got = pool.buffer.cpu().numpy()
    diff = np.nonzero(got != ref)[0]
    assert diff.size == 0, f"{diff.size} bytes differ, first at {diff[:8]}"
    assert_guard_intact(pool.guard, "pool")
