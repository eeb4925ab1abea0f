"""Pins for the oracle's extend (chunked-prefill) attention over an FP8
prefix plus an FP8 chunk ("SGLang's 4-bit KV cache", Figure 2, right-hand
column).

Checked against torch's scaled_dot_product_attention (causal flag with no
prefix; a boolean mask otherwise), a brute-force scalar expansion, closed
forms (equal keys give the mean of the visible values; a dominant key gives
its value) and the invariance of moving chunk tokens into the prefix.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import formats as F
from workloads import f32_to_bf16_bits


def make(lens_p, lens_c, Hq, Hkv, D, seed):
    rng = np.random.default_rng(seed)
    TP, TC = int(sum(lens_p)), int(sum(lens_c))
    def codes(n):
        c = rng.integers(0, 256, (n, Hkv, D), dtype=np.uint8)
        return np.where((c & 0x7F) == 0x7F, c ^ 0x01, c).astype(np.uint8)   # no NaN codes
    q = f32_to_bf16_bits(rng.standard_normal((TC, Hq, D)).astype(np.float32))
    return q, codes(TC), codes(TC), codes(TP), codes(TP)


def dec(c, s):
    return F.e4m3_decode(c) * float(np.float32(s))


def test_no_prefix_is_causal_sdpa():
    q, ck, cv, pk, pv = make([0], [37], 4, 2, 64, 1)
    s = np.array([0.01, 0.02], np.float32)
    sm = np.float32(0.125)
    got = A.extend_attention(q, ck, cv, pk, pv, s, [0], [37], sm)
    qq = torch.from_numpy(F.bf16_to_f32(q).astype(np.float64)).permute(1, 0, 2)   # [Hq, T, D]
    kk = torch.from_numpy(dec(ck, s[0])).permute(1, 0, 2).repeat_interleave(2, 0)
    vv = torch.from_numpy(dec(cv, s[1])).permute(1, 0, 2).repeat_interleave(2, 0)
    ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, is_causal=True, scale=float(sm))
    assert np.allclose(got, ref.permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-13)


def test_prefix_is_masked_sdpa():
    Lp, C = 23, 17
    q, ck, cv, pk, pv = make([Lp], [C], 3, 1, 64, 2)
    s = np.array([0.03, 0.5], np.float32)
    sm = np.float32(0.2)
    got = A.extend_attention(q, ck, cv, pk, pv, s, [Lp], [C], sm)
    keys = np.concatenate([dec(pk, s[0]), dec(ck, s[0])])[:, 0]
    vals = np.concatenate([dec(pv, s[1]), dec(cv, s[1])])[:, 0]
    # row i may attend to key k iff k - Lp <= i: the causal band shifted by Lp
    mask = torch.ones(C, Lp + C, dtype=torch.bool).tril(diagonal=Lp)
    for j in range(3):
        qq = torch.from_numpy(F.bf16_to_f32(q[:, j]).astype(np.float64))
        ref = torch.nn.functional.scaled_dot_product_attention(
            qq[None], torch.from_numpy(keys)[None], torch.from_numpy(vals)[None],
            attn_mask=mask[None], scale=float(sm))
        assert np.allclose(got[:, j], ref[0].numpy(), rtol=1e-12, atol=1e-13)


def test_bruteforce_tiny_by_hand():
    Lp, C, D = 3, 2, 4
    q, ck, cv, pk, pv = make([Lp], [C], 2, 1, D, 3)
    s = np.array([0.25, 0.125], np.float32)
    sm = 0.5
    got = A.extend_attention(q, ck, cv, pk, pv, s, [Lp], [C], np.float32(sm))
    kf = [[float(F.e4m3_decode(np.uint8(x))) * 0.25 for x in row] for row in
          list(pk[:, 0]) + list(ck[:, 0])]
    vf = [[float(F.e4m3_decode(np.uint8(x))) * 0.125 for x in row] for row in
          list(pv[:, 0]) + list(cv[:, 0])]
    for i in range(C):
        for j in range(2):
            qv = [float(F.bf16_to_f32(q[i, j, d])) for d in range(D)]
            sc = [sm * sum(qv[d] * kf[t][d] for d in range(D)) for t in range(Lp + i + 1)]
            mx = max(sc)
            w = [math.exp(x - mx) for x in sc]
            for d in range(D):
                want = sum(w[t] * vf[t][d] for t in range(len(w))) / sum(w)
                assert abs(got[i, j, d] - want) <= 1e-12 * (1 + abs(want))


def test_equal_keys_give_mean_of_visible_values():
    Lp, C = 5, 9
    q, ck, cv, pk, pv = make([Lp], [C], 2, 1, 16, 4)
    ck[:] = 0x38
    pk[:] = 0x38                     # every key equal: uniform weights
    s = np.array([1.0, 1.0], np.float32)
    got = A.extend_attention(q, ck, cv, pk, pv, s, [Lp], [C], np.float32(0.3))
    vals = np.concatenate([F.e4m3_decode(pv), F.e4m3_decode(cv)])[:, 0]
    for i in range(C):
        want = vals[:Lp + i + 1].mean(axis=0)
        assert np.allclose(got[i, 0], want, rtol=1e-13, atol=1e-13)
        assert np.allclose(got[i, 1], want, rtol=1e-13, atol=1e-13)


def test_dominant_key_selects_its_value():
    Lp, C, D = 4, 3, 8
    q, ck, cv, pk, pv = make([Lp], [C], 1, 1, D, 5)
    q[:] = f32_to_bf16_bits(np.ones((C, 1, D), np.float32))
    pk[:] = 0x00
    ck[:] = 0x00
    pk[2] = 0x7E                     # 448 on every channel: score 448 * D * sm
    got = A.extend_attention(q, ck, cv, pk, pv, np.array([1, 1], np.float32), [Lp], [C],
                             np.float32(1.0))
    for i in range(C):
        assert np.allclose(got[i, 0], F.e4m3_decode(pv[2, 0]), rtol=0, atol=1e-12)


def test_moving_chunk_tokens_into_the_prefix():
    # rows t.. of a (Lp, C) call equal the rows of an (Lp + t, C - t) call
    # whose prefix also holds the first t chunk tokens
    Lp, C, t = 11, 20, 7
    q, ck, cv, pk, pv = make([Lp], [C], 4, 2, 32, 6)
    s = np.array([0.02, 0.07], np.float32)
    sm = np.float32(0.17)
    a = A.extend_attention(q, ck, cv, pk, pv, s, [Lp], [C], sm)
    b = A.extend_attention(q[t:], ck[t:], cv[t:], np.concatenate([pk, ck[:t]]),
                           np.concatenate([pv, cv[:t]]), s, [Lp + t], [C - t], sm)
    assert np.allclose(a[t:], b, rtol=1e-12, atol=1e-14)


def test_batch_offsets_and_row_subset():
    lp, lc = [3, 0, 40], [5, 2, 0]
    q, ck, cv, pk, pv = make(lp, lc, 4, 2, 16, 7)
    s = np.array([0.05, 0.05], np.float32)
    sm = np.float32(0.25)
    full = A.extend_attention(q, ck, cv, pk, pv, s, lp, lc, sm)
    # each request alone gives the same rows
    cp, cc = np.cumsum([0] + lp), np.cumsum([0] + lc)
    for b in range(3):
        one = A.extend_attention(q[cc[b]:cc[b + 1]], ck[cc[b]:cc[b + 1]], cv[cc[b]:cc[b + 1]],
                                 pk[cp[b]:cp[b + 1]], pv[cp[b]:cp[b + 1]], s, [lp[b]], [lc[b]], sm)
        assert np.array_equal(full[cc[b]:cc[b + 1]], one)
    sub = A.extend_attention(q, ck, cv, pk, pv, s, lp, lc, sm, rows=[(6, 3), (0, 0)])
    assert np.array_equal(sub[6, 3], full[6, 3]) and np.array_equal(sub[0, 0], full[0, 0])
    assert np.count_nonzero(np.abs(sub).sum(axis=2)) == 2
