"""The k8v4 variant: FP8 keys, 4-bit values, both rotated by a fixed FP32
Hadamard transform before they are quantised.

Test infrastructure only (see ``oracle/__init__.py``).

"SGLang's 4-bit KV cache", section "Against what this site already
established" (the cache that rotates):
the other 4-bit KV cache of the month stores keys in FP8 and values in
4 bits, and applies one fixed FP32 Hadamard rotation of size D to both
operands; an orthogonal rotation spreads a vector's energy over all of its
coordinates, so no single outlier sets the scale.  The page gives no byte
layout and no value encoder; the readings here:

* Rotation: H = S_D / sqrt(D), S_D the Sylvester Hadamard matrix of order D
  (D a power of two); H is symmetric and orthogonal, so H H = I.  On the
  write path it is evaluated in FP32 as the fast Walsh-Hadamard transform:
  stages len = 1, 2, 4, ..., D/2, each replacing the pair (x_i, x_{i+len})
  (i with bit len clear) by (x_i + x_{i+len}, x_i - x_{i+len}), rounded to
  FP32, then one FP32 multiply by float32(1 / sqrt(D)).
* Keys: FP8 E4M3 per tensor, code = E4M3(k_rot / s_K) (the FP8 format of
  ``quant.fp8_quantize``).
* Values: INT4 per (token, head) row, s = amax / 7, code = clamp(rne(v_rot /
  s), -8, 7) (the INT4 format of ``quant.int4_quantize``).
* Layout, one (page, kv head) chunk of P tokens:
  [K codes P*D][V codes P*D/2][V scales FP32 * P]; K codes and V scales in
  rows per token, V codes in token-pair rows by 16-bit halves as in the
  INT4 pool (word k of pair row p, D bytes, holds elements 4k .. 4k+3 of
  token 2p in its low half and of token 2p+1 in its high half).
* Decode: q is rotated too (q_rot = H q), so q_rot . k_rot = q . k before
  quantisation; the output is o = H (sum_t p_t v_hat_rot_t).  In float64.

Parity unpinned for the value encoder and the chunk layout (readings the
page does not fix); every function below is pinned against something other
than itself in ``tests/test_oracle_k8v4.py``.
"""
import numpy as np

from .formats import bf16_to_f32, e4m3_decode
from .quant import _unpack_nibbles, fp8_quantize, int4_quantize


def hadamard_matrix(D):
    """S_D / sqrt(D) in float64, by Sylvester's doubling [[S, S], [S, -S]]."""
    assert D >= 1 and D & (D - 1) == 0
    S = np.ones((1, 1))
    while S.shape[0] < D:
        S = np.block([[S, S], [S, -S]])
    return S / np.sqrt(D)


def fwht_f32(x):
    """FP32 fast Walsh-Hadamard transform along the last axis, scaled by
    float32(1 / sqrt(D)): the write path's rotation, stage by stage."""
    y = np.array(x, dtype=np.float32, copy=True)
    D = y.shape[-1]
    assert D & (D - 1) == 0
    lead = y.shape[:-1]
    n = 1
    while n < D:
        z = y.reshape(lead + (D // (2 * n), 2, n))
        a, b = z[..., 0, :].copy(), z[..., 1, :].copy()
        z[..., 0, :] = (a + b).astype(np.float32)
        z[..., 1, :] = (a - b).astype(np.float32)
        y = z.reshape(lead + (D,))
        n *= 2
    return (y * np.float32(1.0 / np.sqrt(D))).astype(np.float32)


def chunk_bytes(P, D):
    return P * (D + D // 2 + 4)


def new_pool(num_pages, P, Hkv, D, fill=0):
    return np.full(num_pages * Hkv * chunk_bytes(P, D), fill, dtype=np.uint8)


def _chunk(pool, P, Hkv, D, page, head):
    off = (int(page) * Hkv + int(head)) * chunk_bytes(P, D)
    return pool[off:off + chunk_bytes(P, D)]


def _v_code_index(P, D, off):
    """Chunk byte indices [D/2] of token off's packed V codes (byte 2k + j of
    its packed row at 4k + 2 (off % 2) + j of pair row off // 2)."""
    j = np.arange(D // 2)
    return P * D + (off // 2) * D + 2 * (off % 2) + 4 * (j // 2) + (j % 2)


def write(pool, P, Hkv, k_bf16, v_bf16, slot_mapping, s_k):
    """Rotate and quantise T tokens of bf16 K / V ([T, Hkv, D] bit patterns)
    into the pool at slot_mapping (int64 [T]; slots < 0 skipped)."""
    k_bf16, v_bf16 = np.asarray(k_bf16), np.asarray(v_bf16)
    D = k_bf16.shape[-1]
    k_rot = fwht_f32(bf16_to_f32(k_bf16))
    v_rot = fwht_f32(bf16_to_f32(v_bf16))
    kc = fp8_quantize(k_rot, np.float32(s_k))
    vc, vs = int4_quantize(v_rot)
    for t, slot in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        if slot < 0:
            continue
        page, off = divmod(int(slot), P)
        for h in range(Hkv):
            c = _chunk(pool, P, Hkv, D, page, h)
            c[off * D:(off + 1) * D] = kc[t, h]
            c[_v_code_index(P, D, off)] = vc[t, h]
            c[P * D + P * (D // 2) + 4 * off:P * D + P * (D // 2) + 4 * off + 4] = \
                np.asarray([vs[t, h]], np.float32).view(np.uint8)
    return pool


def read_rows(pool, P, Hkv, D, s_k, block_table_row, n, head):
    """Dequantised rotated rows (float64 [n, D]) of K and V for the first n
    tokens of one request and kv head."""
    K = np.zeros((n, D))
    V = np.zeros((n, D))
    for t in range(n):
        page = int(block_table_row[t // P])
        off = t % P
        c = _chunk(pool, P, Hkv, D, page, head)
        K[t] = e4m3_decode(c[off * D:(off + 1) * D]) * np.float64(np.float32(s_k))
        code = _unpack_nibbles(c[_v_code_index(P, D, off)]).astype(np.int64)
        code = np.where(code >= 8, code - 16, code)
        s = c[P * D + P * (D // 2) + 4 * off:P * D + P * (D // 2) + 4 * off + 4].view(np.float32)[0]
        V[t] = code * np.float64(s)
    return K, V


def decode_attention(q_bf16, pool, P, Hkv, s_k, block_table, seq_lens, sm_scale):
    """FP64 decode attention of the k8v4 cache: q_rot = H q, scores over the
    dequantised rotated keys, o = H (sum_t p_t v_rot_t).  q: uint16 bf16 bits
    [B, Hq, D].  Returns float64 [B, Hq, D] (zero rows for empty requests)."""
    q = bf16_to_f32(np.asarray(q_bf16)).astype(np.float64)
    B, Hq, D = q.shape
    G = Hq // Hkv
    H = hadamard_matrix(D)
    out = np.zeros((B, Hq, D))
    for b in range(B):
        n = int(seq_lens[b])
        if n == 0:
            continue
        for h in range(Hkv):
            K, V = read_rows(pool, P, Hkv, D, s_k, block_table[b], n, h)
            for j in range(h * G, (h + 1) * G):
                s = float(sm_scale) * (K @ (H @ q[b, j]))
                p = np.exp(s - s.max())
                out[b, j] = H @ ((p @ V) / p.sum())
    return out
