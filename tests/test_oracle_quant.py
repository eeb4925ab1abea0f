"""Pins for the oracle's NVFP4 / INT4 encoders and pool layout.

Checked against the byte counts the pages print (tests/golden), exact round
trips of representable values, brute-force nearest-value search, Python's
own round-half-even, and the block locality the pages describe.
"""
import os

import numpy as np
import pytest

from oracle import formats as F
from oracle import pool as P
from oracle import quant as Q
from workloads import f32_to_bf16_bits, global_scale_from_amax

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_numbers.txt")


def golden():
    out = {}
    for line in open(GOLDEN):
        if line.strip() and not line.startswith("#"):
            key, val = line.split()[:2]
            out[key] = float(val)
    return out


def test_byte_accounting_matches_the_pages():
    g = golden()
    D, Pg = int(g["qwen27b_head_dim"]), 64
    spec = P.PoolSpec("nvfp4", 1, Pg, 1, D)
    bytes_per_value = spec.chunk_bytes / (Pg * 2 * D)
    assert bytes_per_value == g["nvfp4_fraction_of_fp8"]            # FP8 stores 1 byte/value
    assert round(1 / bytes_per_value, 4) == g["nvfp4_capacity_ratio"]
    # block size from (4 + 8/B)/8 = 0.5625
    assert (8 * g["nvfp4_fraction_of_fp8"] - 4) ** -1 * 8 == g["nvfp4_block_size"] == Q.NVFP4_BLOCK
    layers, heads = int(g["qwen27b_full_attn_layers"]), int(g["qwen27b_kv_heads"])
    elems = layers * heads * D * 2
    assert elems == g["qwen27b_elems_per_token"] == g["qwen27b_fp8_bytes_per_token"]
    per_token = layers * P.PoolSpec("nvfp4", 1, Pg, heads, D).pool_bytes // Pg
    assert per_token == g["qwen27b_nvfp4_bytes_per_token"]
    # INT4 per token and head, and the two page sizes
    i4 = P.PoolSpec("int4", 1, 800, 1, 256)
    assert i4.chunk_bytes / 800 == g["int4_bytes_per_head_token"]
    assert i4.chunk_bytes == g["int4_page_bytes_800"]
    assert P.PoolSpec("int4", 1, 1600, 1, 256).chunk_bytes == g["int4_page_bytes_1600"]
    # the Mamba state does not fit an 800-token page but fits a 1600-token one
    assert g["int4_page_bytes_800"] < g["mamba_state_bytes"] <= g["int4_page_bytes_1600"]


def test_regions_are_16_byte_aligned():
    for fmt in ("nvfp4", "int4"):
        for D in (64, 128, 256):
            for Pg in (16, 64, 256, 1600):
                s = P.PoolSpec(fmt, 2, Pg, 3, D)
                for r in ("kc", "vc", "ks", "vs"):
                    assert s.region(r) % 16 == 0
                assert s.chunk_bytes % 16 == 0


def _representable_block(rng, S_code, g, with_max=True):
    codes = rng.integers(0, 16, 16)
    if with_max:
        codes[rng.integers(16)] = 7 | (rng.integers(2) << 3)
    vals = F.e2m1_decode(codes) * F.e4m3_decode(S_code) * float(g)
    return vals, codes


def test_nvfp4_exact_round_trip_of_representable_values():
    rng = np.random.default_rng(0)
    for _ in range(400):
        g = np.float32(2.0 ** rng.integers(-8, 4))
        S = int(rng.integers(8, 0x7F))               # normal E4M3 scales
        vals, codes = _representable_block(rng, S, g)
        x = f32_to_bf16_bits(vals.astype(np.float32))
        assert np.array_equal(F.bf16_to_f32(x).astype(np.float64), vals)   # exact in bf16
        c, s = Q.nvfp4_quantize(x[None], g)
        assert s[0, 0] == S
        # every code comes back, including the sign of zero (0x8 stays 0x8)
        assert np.array_equal(Q._unpack_nibbles(c)[0], codes.astype(np.uint8))
        assert np.array_equal(Q.nvfp4_dequantize(c, s, g)[0], vals)


def test_nvfp4_codes_are_nearest_values_bruteforce():
    rng = np.random.default_rng(1)
    x = f32_to_bf16_bits(rng.standard_normal((64, 256)).astype(np.float32) * 3)
    g = np.float32(0.01)
    c, s = Q.nvfp4_quantize(x, g)
    xf = F.bf16_to_f32(x).astype(np.float64).reshape(64, 16, 16)
    grid2 = F.e2m1_decode(np.arange(8))
    grid4 = F.e4m3_decode(np.arange(0x7F))
    n = Q._unpack_nibbles(c).reshape(64, 16, 16)
    for r in range(64):
        for b in range(16):
            amax = np.abs(xf[r, b]).max()
            sf = float(np.float32(np.float32(amax) / (np.float32(6.0) * g)))
            chosen = F.e4m3_decode(s[r, b])
            assert abs(chosen - sf) <= np.abs(grid4 - sf).min()
            denom = float(np.float32(np.float32(chosen) * g))
            for i in range(16):
                t = float(np.float32(np.float32(xf[r, b, i]) / np.float32(denom)))
                v = abs(F.e2m1_decode(n[r, b, i]))
                assert abs(v - abs(t)) <= np.abs(grid2 - abs(t)).min()
                assert (n[r, b, i] >> 3) == (1 if np.signbit(np.float32(xf[r, b, i])) else 0)


def test_nvfp4_layer_amax_block_uses_full_scale():
    """With g = amax / (6 * 448) the block holding the layer maximum gets
    the largest E4M3 scale and its maximum element the code for 6."""
    rng = np.random.default_rng(2)
    x = f32_to_bf16_bits(rng.standard_normal((8, 64)).astype(np.float32))
    xf = F.bf16_to_f32(x)
    g = global_scale_from_amax(np.abs(xf).max())
    c, s = Q.nvfp4_quantize(x, g)
    r, i = np.unravel_index(np.argmax(np.abs(xf)), xf.shape)
    assert s[r, i // 16] == 0x7E
    assert Q._unpack_nibbles(c)[r, i] & 7 == 7


def test_nvfp4_zero_block_and_tiny_block():
    x = np.zeros((1, 32), np.uint16)
    x[0, 16:] = f32_to_bf16_bits(np.full(16, -1e-30, np.float32))   # rounds to S == 0
    c, s = Q.nvfp4_quantize(x, np.float32(1.0))
    assert s.tolist() == [[0, 0]] and np.all(c == 0)


def test_nvfp4_block_locality():
    """A per-16 scale confines an outlier to its own block ("SGLang's 4-bit
    KV cache", section "Against what this site already established")."""
    rng = np.random.default_rng(3)
    xf = rng.standard_normal((4, 256)).astype(np.float32)
    g = np.float32(0.005)
    c0, s0 = Q.nvfp4_quantize(f32_to_bf16_bits(xf), g)
    xf2 = xf.copy()
    xf2[1, 37] *= 10.0
    c1, s1 = Q.nvfp4_quantize(f32_to_bf16_bits(xf2), g)
    blk = 37 // 16
    diff_s = np.argwhere(s0 != s1)
    assert all((r, b) == (1, blk) for r, b in diff_s)
    n0, n1 = Q._unpack_nibbles(c0), Q._unpack_nibbles(c1)
    diff_c = np.argwhere(n0 != n1)
    assert len(diff_c) > 0 and all(r == 1 and i // 16 == blk for r, i in diff_c)


def test_int4_round_trip_and_ties():
    rng = np.random.default_rng(4)
    for _ in range(200):
        s = 2.0 ** int(rng.integers(-6, 4))
        codes = rng.integers(-7, 8, 256)
        codes[rng.integers(256)] = 7 * (1 if rng.integers(2) else -1)
        x = f32_to_bf16_bits((codes * s).astype(np.float32))
        c, sc = Q.int4_quantize(x[None])
        assert sc[0] == np.float32(s)
        assert np.array_equal(Q.int4_dequantize(c, sc)[0], codes * s)
    # ties go to even, as Python's round() does
    s = 1.0
    vals = np.array([7.0, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 3.49, -6.5, 4.5], np.float32)
    c, sc = Q.int4_quantize(f32_to_bf16_bits(vals)[None])
    got = Q.int4_dequantize(c, sc)[0] / sc[0]
    assert got.tolist() == [float(round(float(v))) for v in vals]
    z, sz = Q.int4_quantize(np.zeros((1, 256), np.uint16))
    assert sz[0] == 0 and np.all(z == 0)


def test_pool_write_places_rows_by_slot():
    """Every code nibble and scale byte lands where the layout says (computed
    here by hand from the documented order) and nothing else changes."""
    rng = np.random.default_rng(5)
    for fmt in ("nvfp4", "int4", "fp8"):
        D, Pg = 64, 16
        spec = P.PoolSpec(fmt, 5, Pg, 2, D)
        T = 20
        k = f32_to_bf16_bits(rng.standard_normal((T, 2, D)).astype(np.float32))
        v = f32_to_bf16_bits(rng.standard_normal((T, 2, D)).astype(np.float32))
        slots = rng.permutation(5 * Pg)[:T].astype(np.int64)
        slots[3] = -1
        pool = P.new_pool(spec, fill=0xAB)
        P.write(pool, spec, k, v, slots, np.array([0.01, 0.02], np.float32))
        W = {"nvfp4": D // 16, "int4": 4, "fp8": 0}[fmt]     # scale bytes per token
        CB = D if fmt == "fp8" else D // 2                   # code bytes per token
        chunk = Pg * 2 * (CB + W)
        reg = {"kc": 0, "vc": Pg * CB, "ks": 2 * Pg * CB, "vs": 2 * Pg * CB + Pg * W}
        written = np.zeros((spec.pool_bytes, 2), bool)    # per nibble
        for t in range(T):
            if slots[t] < 0:
                continue
            page, off = divmod(int(slots[t]), Pg)
            for h in range(2):
                base = (page * 2 + h) * chunk
                for kind, x, gg in (("k", k, 0.01), ("v", v, 0.02)):
                    if fmt == "fp8":
                        # one byte per element, token rows of D bytes, no scale rows
                        cc = Q.fp8_quantize(x[t, h][None], np.float32(gg))[0]
                        for d in range(D):
                            at = base + reg[kind + "c"] + off * D + d
                            assert pool[at] == cc[d]
                            written[at, :] = True
                        continue
                    if fmt == "nvfp4":
                        cc, ss = Q.nvfp4_quantize(x[t, h][None], np.float32(gg))
                        ss = ss[0]
                    else:
                        cc, sc = Q.int4_quantize(x[t, h][None])
                        ss = sc.astype(np.float32).view(np.uint8)
                    nib = np.empty(D, np.uint8)
                    nib[0::2], nib[1::2] = cc[0] & 0xF, cc[0] >> 4
                    if kind == "v" and fmt == "nvfp4":
                        # pair row off//2 of D bytes; element d in nibble off%2 of byte d
                        for d in range(D):
                            at = base + reg["vc"] + (off // 2) * D + d
                            assert (pool[at] >> (4 * (off % 2))) & 0xF == nib[d]
                            written[at, off % 2] = True
                        for blk in range(W):
                            at = base + reg["vs"] + (off // 2) * 2 * W + 2 * blk + off % 2
                            assert pool[at] == ss[blk]
                            written[at, :] = True
                    else:
                        for d in range(D):
                            if kind == "v":
                                # INT4 V: pair row off//2 of D bytes; word d//4 holds
                                # elements 4k..4k+3 of token 2p in its low 16 bits and
                                # of token 2p+1 in its high 16 bits, element 4k+i in
                                # nibble i of the half
                                at = base + reg["vc"] + (off // 2) * D + 4 * (d // 4) + 2 * (off % 2) + (d % 4) // 2
                            else:
                                at = base + reg[kind + "c"] + off * (D // 2) + d // 2
                            assert (pool[at] >> (4 * (d % 2))) & 0xF == nib[d]
                            written[at, d % 2] = True
                        for i in range(W):
                            at = base + reg[kind + "s"] + off * W + i
                            assert pool[at] == ss[i]
                            written[at, :] = True
        lo_ok = (pool & 0xF) == 0xB
        hi_ok = (pool >> 4) == 0xA
        assert np.all(lo_ok | written[:, 0]) and np.all(hi_ok | written[:, 1])   # nothing else touched


def test_fp8_quantize_matches_torch_cast():
    """FP8 per tensor: E4M3(float32(x) / s), checked against torch's float32 ->
    float8_e4m3fn cast of the same FP32 quotient (in range), the saturation at
    448 and the sign of zero."""
    import torch
    rng = np.random.default_rng(11)
    x = rng.standard_normal((64, 128)).astype(np.float32) * 3
    xb = f32_to_bf16_bits(x)
    for s in (np.float32(0.01), np.float32(1 / 448), np.float32(0.37)):
        q = (F.bf16_to_f32(xb) / s).astype(np.float32)
        keep = np.abs(q) <= 448
        got = Q.fp8_quantize(xb, s)
        want = torch.from_numpy(np.where(keep, q, 0).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(got[keep], want[keep])
        # beyond 448 the code saturates to +-448 (0x7E / 0xFE), never NaN
        over = ~keep
        assert np.all((got[over] & 0x7F) == 0x7E)
        assert np.array_equal(got[over] >> 7, (q[over] < 0).astype(np.uint8))
    # a tiny negative element keeps its sign as -0
    tiny = f32_to_bf16_bits(np.array([[-1e-30, 1e-30, 0.0]], np.float32))
    assert Q.fp8_quantize(tiny, np.float32(1.0)).tolist() == [[0x80, 0x00, 0x00]]
    # decode is code value times s
    c = np.arange(256, dtype=np.uint8)
    finite = (c & 0x7F) != 0x7F
    v = Q.fp8_dequantize(c[finite], np.float32(0.5))
    assert np.allclose(v, torch.from_numpy(c[finite]).view(torch.float8_e4m3fn).float().numpy() * 0.5)


def test_calibrate_global_scale():
    """g = amax / (6 * 448) in FP32, 1 for an all-zero tensor; the layer
    amax then encodes to the largest E4M3 scale (0x7E) and E2M1 code 6."""
    rng = np.random.default_rng(21)
    x = rng.standard_normal((300, 4, 64)).astype(np.float32) * 7
    xb = f32_to_bf16_bits(x)
    amax = np.abs(F.bf16_to_f32(xb)).max()
    g = Q.calibrate_global_scale(xb)
    assert g == np.float32(np.float32(amax) / np.float32(2688.0))
    assert Q.calibrate_global_scale(np.zeros((3, 64), np.uint16)) == np.float32(1.0)
    assert Q.calibrate_global_scale(f32_to_bf16_bits(np.array([[2688.0, -1.0]], np.float32))) == 1.0
    # with the calibrated g the block holding the amax gets scale code 0x7E
    flat = xb.reshape(-1, 64)
    row = np.argmax(np.abs(F.bf16_to_f32(flat)).max(axis=1))
    codes, scales = Q.nvfp4_quantize(flat[row][None], g)
    blk = np.argmax(np.abs(F.bf16_to_f32(flat[row])).reshape(4, 16).max(axis=1))
    assert scales[0, blk] == 0x7E


def test_fp8_input_values_match_torch_cast():
    """The FP8-input write's values: torch's float8_e4m3fn -> float32 cast of
    every code, times the scale in float32."""
    import torch
    codes = np.arange(256, dtype=np.uint8)
    codes = codes[(codes & 0x7F) != 0x7F]                      # no NaN codes
    for s in (np.float32(1.0), np.float32(0.0123), np.float32(3.7)):
        got = Q.fp8_input_values(codes, s)
        want = (torch.from_numpy(codes).view(torch.float8_e4m3fn).float() * float(s)).numpy()
        assert got.dtype == np.float32 and np.array_equal(got, want.astype(np.float32))


@pytest.mark.parametrize("fmt", ["nvfp4", "int4", "fp8"])
def test_write_fp8_equals_write_of_the_same_bf16_values(fmt):
    """With a power-of-two input scale every e4m3(code) * s is a bf16 value,
    so the FP8-input write must store exactly what the bf16 write stores for
    those values (ties the new path to the pinned one)."""
    from oracle import pool as P
    rng = np.random.default_rng(31)
    T, H, D, Pg = 40, 2, 64, 16
    kc = rng.integers(0, 256, (T, H, D), dtype=np.uint8)
    vc = rng.integers(0, 256, (T, H, D), dtype=np.uint8)
    kc = np.where((kc & 0x7F) == 0x7F, kc ^ 1, kc).astype(np.uint8)
    vc = np.where((vc & 0x7F) == 0x7F, vc ^ 1, vc).astype(np.uint8)
    s_in = np.array([0.25, 2.0], np.float32)
    spec = P.PoolSpec(fmt, 4, Pg, H, D)
    slots = rng.permutation(4 * Pg)[:T].astype(np.int64)
    g = np.array([0.01, 0.02], np.float32)
    a = P.write_fp8(P.new_pool(spec), spec, kc, vc, s_in, slots, g)
    kb = f32_to_bf16_bits(Q.fp8_input_values(kc, s_in[0]))
    vb = f32_to_bf16_bits(Q.fp8_input_values(vc, s_in[1]))
    assert np.array_equal(F.bf16_to_f32(kb), Q.fp8_input_values(kc, s_in[0]))   # exact in bf16
    b = P.write(P.new_pool(spec), spec, kb, vb, slots, g)
    assert np.array_equal(a, b)
