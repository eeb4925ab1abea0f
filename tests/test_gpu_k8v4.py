"""GPU parity of the k8v4 variant (FP8 keys, INT4 values, one fixed Hadamard
rotation of both; "SGLang's 4-bit KV cache", section "Against what this site
already established") against the oracle: the write byte for byte, the
decode within the attention gate (max-abs 2e-3, cosine 0.9999) on pools the
oracle wrote."""
import numpy as np
import pytest
import torch

import bit_paged_kv_kv4_gb300 as K
from kv4_testlib import assert_guard_intact, check_close, dev_bf16, guarded_pool
from oracle import k8v4 as KV
from workloads import f32_to_bf16_bits

pytestmark = pytest.mark.gpu


def draws(T, H, D, seed, outlier=7, scale=12.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((2, T, H, D)).astype(np.float32)
    x[:, :, :, outlier % D] *= scale
    return f32_to_bf16_bits(x[0]), f32_to_bf16_bits(x[1])


@pytest.mark.parametrize("D", [64, 128, 256])
def test_k8v4_write_bit_exact(D):
    T, H, P, pages = 300, 2, 16, 24
    k, v = draws(T, H, D, D)
    rng = np.random.default_rng(D + 1)
    slots = rng.permutation(pages * P)[:T].astype(np.int64)
    slots[::13] = -1
    s_k = np.float32(0.05)
    pool = guarded_pool("k8v4", pages, P, H, D, fill=0xA5)
    K.kv4_k8v4_write(dev_bf16(k), dev_bf16(v), torch.from_numpy(slots).cuda(), pool,
                     torch.tensor([s_k], dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()
    assert K.kv4_device_error() == 0
    assert_guard_intact(pool.guard, "pool")
    ref = KV.write(KV.new_pool(pages, P, H, D, fill=0xA5), P, H, k, v, slots, s_k)
    got = pool.buffer.cpu().numpy()
    diff = np.nonzero(got != ref)[0]
    assert diff.size == 0, f"{diff.size} bytes differ, first at {diff[:8]}"


@pytest.mark.parametrize("D", [64, 128, 256])
def test_k8v4_write_many_groups_per_cta(D):
    # more row groups (8 warps of 32 / (D / 32) rows) than the resident grid
    # has CTAs: each CTA loops over several, the next group's input in
    # flight; a ragged last group
    H, P = 4, 16
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    group = 8 * (32 // (D // 32))
    T = 3 * (3 * sms // 2) * group // H + 7
    pages = (T + P - 1) // P + 3
    k, v = draws(T, H, D, D + 5, outlier=D // 3)
    rng = np.random.default_rng(D + 6)
    slots = rng.permutation(pages * P)[:T].astype(np.int64)
    slots[::29] = -1
    s_k = np.float32(0.04)
    pool = guarded_pool("k8v4", pages, P, H, D, fill=0x3C)
    K.kv4_k8v4_write(dev_bf16(k), dev_bf16(v), torch.from_numpy(slots).cuda(), pool,
                     torch.tensor([s_k], dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()
    assert K.kv4_device_error() == 0
    assert_guard_intact(pool.guard, "pool")
    ref = KV.write(KV.new_pool(pages, P, H, D, fill=0x3C), P, H, k, v, slots, s_k)
    got = pool.buffer.cpu().numpy()
    diff = np.nonzero(got != ref)[0]
    assert diff.size == 0, f"{diff.size} bytes differ, first at {diff[:8]}"


@pytest.mark.parametrize("D", [64, 128, 256])
def test_k8v4_write_signed_zeros(D):
    # rows of +0, -0, +x and -x: the rotation makes exact zeros of both
    # signs (-0 + -0 = -0, x + -x = +0), so the FP8 keys' sign of zero and
    # the quotients of zero are checked; all-(+0) and all-(-0) rows too
    H, P, T = 2, 16, 64
    rng = np.random.default_rng(D + 9)
    choices = np.array([0x0000, 0x8000, 0x3FC0, 0xBFC0], np.uint16)   # +0, -0, 1.5, -1.5
    k = choices[rng.integers(0, 4, (T, H, D))]
    v = choices[rng.integers(0, 4, (T, H, D))]
    k[0], v[0] = 0x0000, 0x0000
    k[1], v[1] = 0x8000, 0x8000
    k[2, :, ::2], v[2, :, ::2] = 0x8000, 0x8000                         # -0 and +0 alternating
    k[2, :, 1::2], v[2, :, 1::2] = 0x0000, 0x0000
    slots = np.arange(T, dtype=np.int64)
    s_k = np.float32(0.01)
    pages = (T + P - 1) // P
    pool = guarded_pool("k8v4", pages, P, H, D, fill=0x77)
    K.kv4_k8v4_write(dev_bf16(k), dev_bf16(v), torch.from_numpy(slots).cuda(), pool,
                     torch.tensor([s_k], dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()
    assert K.kv4_device_error() == 0
    assert_guard_intact(pool.guard, "pool")
    ref = KV.write(KV.new_pool(pages, P, H, D, fill=0x77), P, H, k, v, slots, s_k)
    got = pool.buffer.cpu().numpy()
    diff = np.nonzero(got != ref)[0]
    assert diff.size == 0, f"{diff.size} bytes differ, first at {diff[:8]}"
    # the case holds both signs of zero among the FP8 key codes
    kc = ref.reshape(pages, H, -1)[:, :, :P * D].reshape(-1)
    assert (kc == 0x80).any() and (kc == 0x00).any()


def oracle_case(Hkv, Hq, D, lens, P, seed):
    rng = np.random.default_rng(seed)
    B = len(lens)
    need = [(L + P - 1) // P for L in lens]
    num_pages = sum(need) + 2
    perm = rng.permutation(num_pages)
    table = np.full((B, max(max(need), 1)), -1, np.int32)
    at = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[at:at + n]
        at += n
    s_k = np.float32(0.03)
    pool = KV.new_pool(num_pages, P, Hkv, D)
    for b, L in enumerate(lens):
        k, v = draws(L, Hkv, D, seed + 10 + b)
        pos = np.arange(L)
        KV.write(pool, P, Hkv, k, v, table[b, pos // P].astype(np.int64) * P + pos % P, s_k)
    q = f32_to_bf16_bits(rng.standard_normal((B, Hq, D)).astype(np.float32))
    return pool, num_pages, table, np.array(lens, np.int32), s_k, q


def run_decode(pool_np, num_pages, P, Hkv, D, table, lens, s_k, q, chunks, out_dtype=torch.float32):
    pool = K.Pool("k8v4", num_pages, P, Hkv, D, device="cuda")
    pool.buffer.copy_(torch.from_numpy(pool_np))
    B, Hq = q.shape[0], q.shape[1]
    out = torch.full((B, Hq, D), 7.0, dtype=out_dtype, device="cuda")
    ws = torch.empty(max(K.kv4_k8v4_workspace_bytes(B, Hkv, D, chunks), 1), dtype=torch.uint8, device="cuda")
    K.kv4_k8v4_decode_attention(dev_bf16(q), pool, torch.tensor([s_k], device="cuda"),
                                torch.from_numpy(table).cuda(), torch.from_numpy(lens).cuda(),
                                np.float32(1.0 / np.sqrt(D)), out, chunks, ws)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("D,Hkv,Hq,lens,chunks", [
    (64, 2, 6, [37, 300, 0, 1], 1),
    (64, 2, 6, [37, 300, 0, 1], 5),
    (128, 1, 8, [700], 3),
    (256, 4, 24, [1000, 2500, 17], 4),
])
def test_k8v4_decode_matches_oracle(D, Hkv, Hq, lens, chunks):
    P = 16
    pool, num_pages, table, lens, s_k, q = oracle_case(Hkv, Hq, D, lens, P, D + chunks)
    got = run_decode(pool, num_pages, P, Hkv, D, table, lens, s_k, q, chunks).cpu().numpy()
    assert K.kv4_device_error() == 0
    want = KV.decode_attention(q, pool, P, Hkv, s_k, table, lens, np.float32(1.0 / np.sqrt(D)))
    for b in range(len(lens)):
        if lens[b] == 0:
            assert not got[b].any()
    check_close(got, want, what=f"k8v4 D{D}")


def test_k8v4_bf16_output_and_chunk_count_consistency():
    D, Hkv, Hq, P = 256, 2, 12, 16
    pool, num_pages, table, lens, s_k, q = oracle_case(Hkv, Hq, D, [900, 64], P, 9)
    a = run_decode(pool, num_pages, P, Hkv, D, table, lens, s_k, q, 1).cpu().numpy()
    b = run_decode(pool, num_pages, P, Hkv, D, table, lens, s_k, q, 7).cpu().numpy()
    assert np.abs(a - b).max() <= 1e-4                         # merging order only
    h = run_decode(pool, num_pages, P, Hkv, D, table, lens, s_k, q, 7, torch.bfloat16).float().cpu().numpy()
    assert np.all(np.abs(h - b) <= np.abs(b) * 2.0 ** -8 + 1e-30)


def test_k8v4_bad_table_entry_is_flagged():
    D, Hkv, Hq, P = 64, 1, 2, 16
    pool, num_pages, table, lens, s_k, q = oracle_case(Hkv, Hq, D, [40], P, 3)
    table = table.copy()
    table[0, 1] = num_pages + 5                                # outside the pool
    run_decode(pool, num_pages, P, Hkv, D, table, lens, s_k, q, 2)
    assert K.kv4_device_error() == 4                           # KV4_EBOUNDS
