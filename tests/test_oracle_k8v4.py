"""Pins for the oracle's k8v4 variant (FP8 keys, 4-bit values, one fixed
Hadamard rotation of both; "SGLang's 4-bit KV cache", section "Against what
this site already established").

The rotation against scipy's Hadamard matrix and against closed forms (an
outlier spread over every coordinate, orthogonality), and the decode against
the same attention computed the other way round: keys and values rotated
back instead of the query rotated forward.
"""
import numpy as np
import pytest
import scipy.linalg

from oracle import k8v4 as KV
from oracle import quant as Q
from oracle import formats as F
from workloads import f32_to_bf16_bits


@pytest.mark.parametrize("D", [64, 128, 256])
def test_hadamard_matrix_is_scipy_sylvester_and_orthogonal(D):
    H = KV.hadamard_matrix(D)
    assert np.array_equal(H * np.sqrt(D), scipy.linalg.hadamard(D))
    assert np.allclose(H @ H, np.eye(D), atol=1e-12) and np.array_equal(H, H.T)


@pytest.mark.parametrize("D", [64, 256])
def test_fwht_exact_on_small_integers(D):
    # integer inputs keep every butterfly sum exact in FP32, and 1/sqrt(D) is a
    # power of two at D = 64 and 256, so the FP32 transform is exact
    rng = np.random.default_rng(D)
    x = rng.integers(-50, 50, (7, D)).astype(np.float32)
    assert np.array_equal(KV.fwht_f32(x).astype(np.float64), x.astype(np.float64) @ KV.hadamard_matrix(D))


def test_fwht_close_to_fp64_matrix_and_an_involution():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((20, 128)) * 3).astype(np.float32)
    y = KV.fwht_f32(x)
    ref = x.astype(np.float64) @ KV.hadamard_matrix(128)
    assert np.max(np.abs(y - ref)) <= 1e-5 * np.max(np.abs(ref))
    assert np.allclose(KV.fwht_f32(y), x, rtol=0, atol=1e-4)


def test_rotation_spreads_one_outlier_over_every_coordinate():
    x = np.zeros((1, 256), np.float32)
    x[0, 77] = 48.0
    y = KV.fwht_f32(x)
    assert np.all(np.abs(y) == np.float32(3.0))              # 48 / sqrt(256) everywhere


def build(Hkv, D, lens, P, seed, Hq):
    rng = np.random.default_rng(seed)
    B = len(lens)
    pages = [(L + P - 1) // P for L in lens]
    num_pages = sum(pages) + 1
    perm = rng.permutation(num_pages)
    table = np.full((B, max(max(pages), 1)), -1, np.int64)
    at = 0
    for b, n in enumerate(pages):
        table[b, :n] = perm[at:at + n]
        at += n
    pool = KV.new_pool(num_pages, P, Hkv, D)
    s_k = np.float32(0.02)
    for b, L in enumerate(lens):
        x = rng.standard_normal((2, L, Hkv, D)).astype(np.float32)
        x[:, :, :, 5] *= 8                                    # an outlier channel
        pos = np.arange(L)
        slots = table[b, pos // P] * P + pos % P
        KV.write(pool, P, Hkv, f32_to_bf16_bits(x[0]), f32_to_bf16_bits(x[1]), slots, s_k)
    q = f32_to_bf16_bits(rng.standard_normal((B, Hq, D)).astype(np.float32))
    return pool, table, np.array(lens), q, s_k


def test_decode_equals_attention_over_rotated_back_keys_and_values():
    Hkv, D, P, Hq = 2, 64, 16, 6
    pool, table, lens, q, s_k = build(Hkv, D, [37, 70, 0], P, 3, Hq)
    sm = 0.125
    got = KV.decode_attention(q, pool, P, Hkv, s_k, table, lens, sm)
    H = KV.hadamard_matrix(D)
    G = Hq // Hkv
    for b in range(3):
        if lens[b] == 0:
            assert not got[b].any()
            continue
        for h in range(Hkv):
            K, V = KV.read_rows(pool, P, Hkv, D, s_k, table[b], int(lens[b]), h)
            Kb, Vb = K @ H, V @ H                              # back to the unrotated basis
            for j in range(h * G, (h + 1) * G):
                qv = F.bf16_to_f32(q[b, j]).astype(np.float64)
                s = sm * (Kb @ qv)
                p = np.exp(s - s.max())
                assert np.allclose(got[b, j], (p @ Vb) / p.sum(), rtol=1e-11, atol=1e-12)


def test_write_stores_the_rotated_codes_in_their_rows():
    Hkv, D, P = 1, 64, 16
    pool = KV.new_pool(2, P, Hkv, D, fill=0xEE)
    rng = np.random.default_rng(5)
    k = f32_to_bf16_bits(rng.standard_normal((3, 1, D)).astype(np.float32))
    v = f32_to_bf16_bits(rng.standard_normal((3, 1, D)).astype(np.float32))
    KV.write(pool, P, Hkv, k, v, np.array([17, -1, 2]), np.float32(0.05))
    c1 = pool[KV.chunk_bytes(P, D):]                          # page 1 (slot 17 -> offset 1)
    assert np.array_equal(c1[D:2 * D], Q.fp8_quantize(KV.fwht_f32(F.bf16_to_f32(k[0])), np.float32(0.05))[0])
    vc, vs = Q.int4_quantize(KV.fwht_f32(F.bf16_to_f32(v[2])))
    c0 = pool[:KV.chunk_bytes(P, D)]
    # slot 2: pair row 1 of the V codes, the even token's low 16-bit halves
    pair = c0[P * D + 1 * D:P * D + 2 * D]
    assert np.array_equal(pair.reshape(-1, 4)[:, :2].reshape(-1), vc[0])
    assert np.all(pair.reshape(-1, 4)[:, 2:] == 0xEE)             # the odd token's halves untouched
    assert c0[P * D + P * (D // 2) + 8:P * D + P * (D // 2) + 12].view(np.float32)[0] == vs[0]
    assert np.all(c0[:2 * D] == 0xEE) and np.all(c1[:D] == 0xEE)   # untouched rows
