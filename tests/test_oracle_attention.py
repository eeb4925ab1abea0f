"""Pins for the oracle's attention, split-KV combine and prefix dequant.

Checked against hand expansion with Python loops, closed-form special cases
(equal keys, one dominant key), invariances the definition implies (page
size, page permutation, split count), torch's scaled_dot_product_attention,
and torch's float8 cast for the FP8 workspace.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import formats as F
from oracle import pool as P
from oracle import quant as Q
from workloads import f32_to_bf16_bits, global_scale_from_amax


def build(fmt, Hkv, D, lens, page, seed=0, Hq=None, perm=True, kv=None):
    """Pool + tables for random bf16 K/V written through the oracle."""
    rng = np.random.default_rng(seed)
    B = len(lens)
    need = [(L + page - 1) // page for L in lens]
    num_pages = sum(need) + 2
    order = np.random.default_rng(seed + 1000).permutation(num_pages) if perm else np.arange(num_pages)
    maxp = max(max(need), 1)
    table = np.full((B, maxp), -1, np.int32)
    at = 0
    for b, n in enumerate(need):
        table[b, :n] = order[at:at + n]
        at += n
    spec = P.PoolSpec(fmt, num_pages, page, Hkv, D)
    pool = P.new_pool(spec)
    Ks, Vs = [], []
    for b, L in enumerate(lens):
        if kv is None:
            k = f32_to_bf16_bits(rng.standard_normal((L, Hkv, D)).astype(np.float32))
            v = f32_to_bf16_bits(rng.standard_normal((L, Hkv, D)).astype(np.float32))
        else:
            k, v = kv(b, L)
        Ks.append(k)
        Vs.append(v)
    allk = np.concatenate([k.reshape(-1) for k in Ks] + [np.zeros(1, np.uint16)])
    allv = np.concatenate([v.reshape(-1) for v in Vs] + [np.zeros(1, np.uint16)])
    g = np.array([global_scale_from_amax(np.abs(F.bf16_to_f32(allk)).max()),
                  global_scale_from_amax(np.abs(F.bf16_to_f32(allv)).max())], np.float32)
    for b, L in enumerate(lens):
        pos = np.arange(L)
        slots = table[b, pos // page].astype(np.int64) * page + pos % page
        P.write(pool, spec, Ks[b], Vs[b], slots, g)
    Hq = Hq or Hkv
    q = f32_to_bf16_bits(rng.standard_normal((B, Hq, D)).astype(np.float32))
    return spec, pool, table, np.array(lens, np.int32), g, q, Ks, Vs


def test_bruteforce_tiny_by_hand():
    """D = 16, 3 tokens, pages of 16: expand every step with Python loops."""
    spec, pool, table, lens, g, q, Ks, Vs = build("nvfp4", 1, 16, [3], 16, seed=1, Hq=2)
    sm = np.float32(0.25)
    got = A.decode_attention(q, pool, spec, g, table, lens, sm)
    page = int(table[0, 0])
    base = (page * 1 + 0) * spec.chunk_bytes

    def row(kind, t):
        gg = float(g[0] if kind == "k" else g[1])
        vals = []
        if kind == "k":
            # one row per token: 8 bytes, element 2j low nibble of byte j; 1 scale byte
            cbase = base + spec.region("kc") + t * 8
            s = F.e4m3_decode(pool[base + spec.region("ks") + t])
            for j in range(8):
                byte = int(pool[cbase + j])
                for nib in (byte & 0xF, byte >> 4):
                    vals.append(float(F.e2m1_decode(nib)) * float(s) * gg)
        else:
            # token pairs: byte d of pair row t//2 (16 bytes) holds element d of
            # token t in nibble t%2; the pair's scale row is (s_even, s_odd)
            cbase = base + spec.region("vc") + (t // 2) * 16
            s = F.e4m3_decode(pool[base + spec.region("vs") + (t // 2) * 2 + (t % 2)])
            for d in range(16):
                nib = (int(pool[cbase + d]) >> (4 * (t % 2))) & 0xF
                vals.append(float(F.e2m1_decode(nib)) * float(s) * gg)
        return vals

    for j in range(2):
        qq = [float(x) for x in F.bf16_to_f32(q[0, j])]
        sc = [float(sm) * sum(a * b for a, b in zip(qq, row("k", t))) for t in range(3)]
        mx = max(sc)
        w = [math.exp(s - mx) for s in sc]
        out = [sum(w[t] * row("v", t)[d] for t in range(3)) / sum(w) for d in range(16)]
        assert np.allclose(got[0, j], out, rtol=1e-13, atol=1e-15)


def test_equal_keys_give_mean_of_values():
    D, L = 64, 40
    rng = np.random.default_rng(2)
    krow = f32_to_bf16_bits(rng.standard_normal(D).astype(np.float32))

    def kv(b, L):
        k = np.broadcast_to(krow, (L, 1, D)).copy()
        v = f32_to_bf16_bits(rng.standard_normal((L, 1, D)).astype(np.float32))
        return k, v

    spec, pool, table, lens, g, q, Ks, Vs = build("nvfp4", 1, D, [L], 16, kv=kv)
    got = A.decode_attention(q, pool, spec, g, table, lens, np.float32(0.125))
    vh = Q.nvfp4_dequantize(*Q.nvfp4_quantize(Vs[0][:, 0], g[1]), g[1])
    assert np.allclose(got[0, 0], vh.mean(axis=0), rtol=1e-12, atol=1e-14)


def test_dominant_key_selects_its_value():
    D, L = 64, 33
    rng = np.random.default_rng(3)
    qv = rng.standard_normal(D).astype(np.float32)

    def kv(b, L):
        k = f32_to_bf16_bits(0.01 * rng.standard_normal((L, 1, D)).astype(np.float32))
        k[17, 0] = f32_to_bf16_bits(qv * 50)
        v = f32_to_bf16_bits(rng.standard_normal((L, 1, D)).astype(np.float32))
        return k, v

    spec, pool, table, lens, g, q, Ks, Vs = build("nvfp4", 1, D, [L], 16, kv=kv)
    q[0, 0] = f32_to_bf16_bits(qv)
    got = A.decode_attention(q, pool, spec, g, table, lens, np.float32(1.0))
    vh = Q.nvfp4_dequantize(*Q.nvfp4_quantize(Vs[0][17:18, 0], g[1]), g[1])[0]
    assert np.allclose(got[0, 0], vh, rtol=0, atol=1e-12)


@pytest.mark.parametrize("fmt", ["nvfp4", "int4"])
def test_invariant_to_page_size_and_permutation(fmt):
    lens = [50, 1, 130]
    outs = []
    for page, perm in ((16, False), (16, True), (64, True), (32, True)):
        spec, pool, table, L, g, q, Ks, Vs = build(fmt, 2, 64, lens, page, seed=7, Hq=6, perm=perm)
        outs.append(A.decode_attention(q, pool, spec, g, table, L, np.float32(0.125)))
    for o in outs[1:]:
        assert np.allclose(o, outs[0], rtol=1e-12, atol=1e-14)


def test_matches_torch_sdpa_when_group_is_one():
    spec, pool, table, lens, g, q, Ks, Vs = build("nvfp4", 3, 64, [70, 5], 16, seed=8, Hq=3)
    sm = np.float32(0.125)
    got = A.decode_attention(q, pool, spec, g, table, lens, sm)
    for b in range(2):
        for h in range(3):
            kh = Q.nvfp4_dequantize(*Q.nvfp4_quantize(Ks[b][:, h], g[0]), g[0])
            vh = Q.nvfp4_dequantize(*Q.nvfp4_quantize(Vs[b][:, h], g[1]), g[1])
            qq = torch.from_numpy(F.bf16_to_f32(q[b, h]).astype(np.float64))[None, None, None]
            ref = torch.nn.functional.scaled_dot_product_attention(
                qq, torch.from_numpy(kh)[None, None], torch.from_numpy(vh)[None, None],
                scale=float(sm))
            assert np.allclose(got[b, h], ref[0, 0, 0].numpy(), rtol=1e-12, atol=1e-14)


def test_gqa_groups_are_contiguous():
    spec, pool, table, lens, g, q, Ks, Vs = build("nvfp4", 2, 64, [40], 16, seed=9, Hq=4)
    got = A.decode_attention(q, pool, spec, g, table, lens, np.float32(0.125))
    # query heads 0,1 read kv head 0 and 2,3 read kv head 1: swapping the kv
    # heads' data while swapping the query halves leaves the output permuted
    q2 = q[:, [2, 3, 0, 1]]
    spec2, pool2, table2, lens2, g2, _, _, _ = build(
        "nvfp4", 2, 64, [40], 16, seed=9, Hq=4,
        kv=lambda b, L: (Ks[0][:, ::-1].copy(), Vs[0][:, ::-1].copy()))
    got2 = A.decode_attention(q2, pool2, spec2, g2, table2, lens2, np.float32(0.125))
    assert np.allclose(got2[:, [2, 3, 0, 1]], got, rtol=1e-12, atol=1e-14)


def test_empty_sequence_is_zero_and_rows_subset():
    spec, pool, table, lens, g, q, Ks, Vs = build("nvfp4", 1, 64, [0, 20], 16, seed=10, Hq=2)
    full = A.decode_attention(q, pool, spec, g, table, lens, np.float32(0.1))
    assert np.all(full[0] == 0)
    part = A.decode_attention(q, pool, spec, g, table, lens, np.float32(0.1), rows=[(1, 1)])
    assert np.allclose(part[1, 1], full[1, 1], rtol=1e-13, atol=1e-15) and np.isnan(part[1, 0]).all()


def test_lse_combine_equals_full_softmax():
    rng = np.random.default_rng(11)
    for S in (1, 2, 7, 128):
        L = int(rng.integers(S, 3000))
        s = rng.standard_normal(L) * 4
        v = rng.standard_normal((L, 16))
        cuts = np.sort(rng.choice(np.arange(L + 1), S - 1, replace=True))
        bounds = np.concatenate([[0], cuts, [L]])          # empty splits allowed
        m, l, o = A.split_partials(s, v, bounds)
        p = np.exp(s - s.max())
        ref = p @ v / p.sum()
        assert np.allclose(A.lse_combine(m, l, o), ref, rtol=1e-12, atol=1e-14)
    assert np.all(A.lse_combine(np.full(3, -np.inf), np.zeros(3), np.ones((3, 4))) == 0)


@pytest.mark.parametrize("fmt", ["nvfp4", "int4"])
def test_dequant_prefix_vs_torch_float8(fmt):
    spec, pool, table, lens, g, q, Ks, Vs = build(fmt, 2, 64, [37, 80], 16, seed=12)
    prefix = np.array([30, 64], np.int64)
    s8 = np.array([6 * g[0], 6 * g[1]], np.float32) if fmt == "nvfp4" else np.array([0.02, 0.03], np.float32)
    wk, wv = A.dequant_prefix(pool, spec, g, table, prefix, s8)
    assert wk.shape == (94, 2, 64)
    for b, n in enumerate(prefix):
        row0 = 0 if b == 0 else prefix[0]
        for h in range(2):
            for kind, src, ws, gg, ss in (("k", Ks, wk, g[0], s8[0]), ("v", Vs, wv, g[1], s8[1])):
                x = src[b][:n, h]
                if fmt == "nvfp4":
                    c, s = Q.nvfp4_quantize(x, gg)
                    e = torch.from_numpy(F.e2m1_decode(Q._unpack_nibbles(c)).astype(np.float32))
                    sc = torch.from_numpy(F.e4m3_decode(s).astype(np.float32))
                    xh = (e.view(n, -1, 16) * sc[:, :, None]).view(n, -1) * float(gg)
                else:
                    c, s = Q.int4_quantize(x)
                    n_ = Q._unpack_nibbles(c).astype(np.int64)
                    xh = torch.from_numpy(np.where(n_ >= 8, n_ - 16, n_).astype(np.float32)) * \
                        torch.from_numpy(s)[:, None]
                y = xh / float(ss)
                assert float(y.abs().max()) < 464
                ref = y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
                assert np.array_equal(ws[row0:row0 + n, h], ref)


def test_int4_error_within_half_step():
    """INT4 with s = amax / 7 never clamps, so every decoded value lies
    within half a quantisation step of its input (the format's error bound)."""
    rng = np.random.default_rng(13)
    x = f32_to_bf16_bits((rng.standard_normal((500, 256)) * rng.uniform(0.1, 10, (500, 1))).astype(np.float32))
    c, s = Q.int4_quantize(x)
    err = np.abs(Q.int4_dequantize(c, s) - F.bf16_to_f32(x))
    assert np.all(err <= 0.5 * s[:, None] * (1 + 1e-6))
    n = Q._unpack_nibbles(c).astype(np.int64)
    assert np.all((np.where(n >= 8, n - 16, n) >= -7))          # -8 never needed


def test_nvfp4_error_within_half_step_when_unsaturated():
    rng = np.random.default_rng(14)
    x = f32_to_bf16_bits(rng.standard_normal((300, 256)).astype(np.float32))
    g = np.float32(0.003)
    c, s = Q.nvfp4_quantize(x, g)
    xf = F.bf16_to_f32(x).astype(np.float64).reshape(300, 16, 16)
    denom = (F.e4m3_decode(s) * float(g))[..., None]
    t = np.abs(xf) / denom
    err = np.abs(Q.nvfp4_dequantize(c, s, g).reshape(300, 16, 16) - xf) / denom
    step = np.where(t < 2, 0.5, np.where(t < 4, 1.0, 2.0))
    ok = t <= 6
    assert np.all(err[ok] <= 0.5 * step[ok] * (1 + 1e-6))
    assert np.all(err[~ok] <= (t[~ok] - 6) * (1 + 1e-6))


def test_int4_bruteforce_tiny_by_hand():
    """INT4, D = 16, 3 tokens: read every code at the position the layout
    gives (K in token rows; V in token-pair rows by 16-bit halves) with its
    per-token FP32 scale and expand the attention with Python loops."""
    spec, pool, table, lens, g, q, Ks, Vs = build("int4", 1, 16, [3], 16, seed=3, Hq=2)
    sm = np.float32(0.25)
    got = A.decode_attention(q, pool, spec, g, table, lens, sm)
    page = int(table[0, 0])
    base = page * spec.chunk_bytes

    def signed(n):
        return n - 16 if n >= 8 else n

    def row(kind, t):
        s = float(pool[base + spec.region(kind + "s") + 4 * t:base + spec.region(kind + "s") + 4 * t + 4]
                  .view(np.float32)[0])
        vals = []
        for d in range(16):
            if kind == "k":
                byte = int(pool[base + spec.region("kc") + t * 8 + d // 2])
            else:
                # pair row t//2 (16 bytes): word d//4 holds elements 4k..4k+3 of the
                # even token in its low half and of the odd token in its high half
                byte = int(pool[base + spec.region("vc") + (t // 2) * 16 + 4 * (d // 4) + 2 * (t % 2) +
                                (d % 4) // 2])
            vals.append(signed((byte >> (4 * (d % 2))) & 0xF) * s)
        return vals

    for j in range(2):
        qq = [float(x) for x in F.bf16_to_f32(q[0, j])]
        sc = [float(sm) * sum(a * b for a, b in zip(qq, row("k", t))) for t in range(3)]
        mx = max(sc)
        w = [math.exp(x - mx) for x in sc]
        out = [sum(w[t] * row("v", t)[d] for t in range(3)) / sum(w) for d in range(16)]
        assert np.allclose(got[0, j], out, rtol=1e-13, atol=1e-15)


def test_fp8_bruteforce_tiny_by_hand():
    """FP8 pool, D = 16, 3 tokens: read every code byte at the position the
    layout gives (token rows of D bytes), decode it with torch's float8 view
    and expand the attention with Python loops."""
    spec, pool, table, lens, g, q, Ks, Vs = build("fp8", 1, 16, [3], 16, seed=4, Hq=2)
    sm = np.float32(0.25)
    got = A.decode_attention(q, pool, spec, g, table, lens, sm)
    page = int(table[0, 0])
    base = page * spec.chunk_bytes

    def row(kind, t):
        start = base + (0 if kind == "k" else 16 * 16) + t * 16
        vals = torch.from_numpy(pool[start:start + 16].copy()).view(torch.float8_e4m3fn).double().numpy()
        return list(vals * float(g[0] if kind == "k" else g[1]))

    for j in range(2):
        qq = [float(x) for x in F.bf16_to_f32(q[0, j])]
        sc = [float(sm) * sum(a * b for a, b in zip(qq, row("k", t))) for t in range(3)]
        mx = max(sc)
        w = [math.exp(s - mx) for s in sc]
        out = [sum(w[t] * row("v", t)[d] for t in range(3)) / sum(w) for d in range(16)]
        assert np.allclose(got[0, j], out, rtol=1e-13, atol=1e-15)
