"""Seeded synthetic workloads for the 4-bit paged KV cache.

This module only draws inputs: shapes, value distributions, sequence
lengths, page tables and slot mappings.  It holds none of the cache
method's arithmetic, so both the CUDA path and the CPU oracle may use it.

The workloads follow the pages' serving runs (the full-attention layers of
the 27B model, 24 query and 4 KV heads of dimension 256, at 32K / 160K / 1M
context, from
"SGLang's 4-bit KV cache", sections "The 56% survives its own scale" and
"The decode gain, separated"; and the INT4 lane at 220,000 tokens with
1600-token pages from "KV cache in 4 bits").  No dataset, trace or weight is
used: every value is drawn from a seeded generator.

Values are drawn per (request, kv head, 64K-token chunk) from numpy's PCG64
seeded with (workload seed, tag, request, head, chunk), so any slice can be
regenerated on its own.  bf16 values are produced from float32 draws by
round-to-nearest-even on the bit pattern and returned as uint16.
"""
from dataclasses import dataclass, field

import numpy as np

CHUNK = 1 << 16          # tokens per generator chunk
E2M1_MAX, E4M3_MAX = 6.0, 448.0


def f32_to_bf16_bits(x):
    """float32 -> bf16 bit patterns (uint16), round to nearest even (finite
    inputs; uint32 arithmetic cannot overflow below the NaN range)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    u = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return u.astype(np.uint16)


def bf16_bits_to_f32(u16):
    return (np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclass(frozen=True)
class Workload:
    name: str
    fmt: str                 # "nvfp4" or "int4"
    num_kv_heads: int
    num_q_heads: int
    head_dim: int
    batch: int
    page_size: int
    len_lo: int              # sequence lengths uniform in [len_lo, len_hi]
    len_hi: int
    dist: str = "normal"     # "normal" or "student_t4"
    outliers: int = 0        # outlier channels per kv head
    outlier_scale: float = 1.0
    outlier_kv: str = "kv"   # "k": keys only, "kv": keys and values
    seed: int = 0
    num_splits: int = 0      # 0 = library default
    prefix_chunk: int = 0    # chunked-prefill chunk (dequant-prefix workloads)
    notes: str = field(default="", compare=False)

    @property
    def group(self):
        return self.num_q_heads // self.num_kv_heads

    def seq_lens(self):
        rng = np.random.Generator(np.random.PCG64([self.seed, 1]))
        return rng.integers(self.len_lo, self.len_hi + 1, size=self.batch).astype(np.int32)

    def pages_needed(self, seq_lens):
        return [(int(L) + self.page_size - 1) // self.page_size for L in seq_lens]

    def block_table(self, seq_lens, spare_pages=3):
        """(num_pages, block_table int32 [B, max_pages]).  Physical pages are a
        seeded permutation (tables are not contiguous); unused entries are -1."""
        need = self.pages_needed(seq_lens)
        num_pages = sum(need) + spare_pages
        rng = np.random.Generator(np.random.PCG64([self.seed, 2]))
        perm = rng.permutation(num_pages).astype(np.int32)
        max_pages = max(max(need), 1)
        table = np.full((self.batch, max_pages), -1, dtype=np.int32)
        at = 0
        for b, n in enumerate(need):
            table[b, :n] = perm[at:at + n]
            at += n
        return num_pages, table

    def outlier_channels(self, head):
        if self.outliers == 0:
            return np.zeros(0, dtype=np.int64)
        rng = np.random.Generator(np.random.PCG64([self.seed, 3, head]))
        return np.sort(rng.choice(self.head_dim, self.outliers, replace=False))

    def kv_chunk(self, b, h, c, n):
        """K and V bf16 bits [n, D] for tokens [c*CHUNK, c*CHUNK + n) of (b, h)."""
        rng = np.random.Generator(np.random.PCG64([self.seed, 4, b, h, c]))
        shape = (2, n, self.head_dim)
        if self.dist == "student_t4":
            x = rng.standard_t(4.0, size=shape).astype(np.float32)
        else:
            x = rng.standard_normal(size=shape, dtype=np.float32)
        ch = self.outlier_channels(h)
        if ch.size:
            x[0][:, ch] *= np.float32(self.outlier_scale)
            if self.outlier_kv == "kv":
                x[1][:, ch] *= np.float32(self.outlier_scale)
        return f32_to_bf16_bits(x[0]), f32_to_bf16_bits(x[1])

    def kv_request(self, b, h, L):
        """K, V bf16 bits [L, D] of the first L tokens of (b, h)."""
        ks, vs = [], []
        for c in range((L + CHUNK - 1) // CHUNK):
            n = min(CHUNK, L - c * CHUNK)
            k, v = self.kv_chunk(b, h, c, n)
            ks.append(k)
            vs.append(v)
        if not ks:
            z = np.zeros((0, self.head_dim), np.uint16)
            return z, z
        return np.concatenate(ks), np.concatenate(vs)

    def q(self):
        rng = np.random.Generator(np.random.PCG64([self.seed, 5]))
        x = rng.standard_normal(size=(self.batch, self.num_q_heads, self.head_dim), dtype=np.float32)
        return f32_to_bf16_bits(x)

    def sm_scale(self):
        return np.float32(1.0 / np.sqrt(self.head_dim))


# --- device-side draws (large workloads) -----------------------------------------
# At the 32K..1M sizes the host generator above is too slow (billions of
# values), so the same distributions are drawn on the GPU by torch's seeded
# Philox generator, one generator per (workload seed, request).  These are
# inputs only; a test hands the oracle the slices it checks, copied to the host.
def device_kv(w, b, L, device):
    """bf16 [2, L, Hkv, D] (K then V) of request b, drawn on `device`."""
    import torch
    gen = torch.Generator(device=device).manual_seed(1_000_003 * (w.seed + 1) + b)
    shape = (2, L, w.num_kv_heads, w.head_dim)
    x = torch.randn(shape, generator=gen, device=device)
    if w.dist == "student_t4":
        chi = torch.zeros(shape, device=device)
        for _ in range(4):
            chi += torch.randn(shape, generator=gen, device=device) ** 2
        x = x / torch.sqrt(chi / 4.0)
    for h in range(w.num_kv_heads):
        ch = w.outlier_channels(h)
        if ch.size:
            idx = torch.from_numpy(ch).to(device)
            x[0, :, h, idx] *= w.outlier_scale
            if w.outlier_kv == "kv":
                x[1, :, h, idx] *= w.outlier_scale
    return x.to(torch.bfloat16)


def device_q(w, device, salt=0):
    """bf16 [B, Hq, D] queries, plus bf16 [B, Hkv, D] K and V of one new token."""
    import torch
    gen = torch.Generator(device=device).manual_seed(7_000_003 * (w.seed + 1) + salt)
    q = torch.randn((w.batch, w.num_q_heads, w.head_dim), generator=gen, device=device)
    kv = torch.randn((2, w.batch, w.num_kv_heads, w.head_dim), generator=gen, device=device)
    return q.to(torch.bfloat16), kv[0].to(torch.bfloat16), kv[1].to(torch.bfloat16)


def fp8_kv_codes(seed, L, Hkv, D, device, outlier_channels=None, outlier_scale=1.0, scales=None):
    """Seeded FP8 K/V input of the extend path: normal draws (outlier channels
    of each kv head scaled up) mapped onto the E4M3 range by per-tensor scales
    and encoded by torch's float8_e4m3fn cast.  Returns (uint8 codes
    [2, L, Hkv, D], float32 scales [2]); `scales` fixes the scales instead of
    deriving them from the draws' maxima (amax / 448)."""
    import torch
    gen = torch.Generator(device=device).manual_seed(9_000_011 * (seed + 1) + L)
    x = torch.randn((2, L, Hkv, D), generator=gen, device=device)
    if outlier_channels is not None:
        for h, ch in enumerate(outlier_channels):
            if len(ch):
                x[:, :, h, torch.as_tensor(ch, device=device)] *= outlier_scale
    if scales is None:
        am = x.abs().amax(dim=(1, 2, 3)).cpu().numpy() if L else np.ones(2, np.float32)
        scales = np.array([fp8_scale_from_amax(a) for a in am], np.float32)
    s = torch.as_tensor(np.asarray(scales, np.float32), device=device)
    # saturate like a satfinite encoder: fixed scales may not cover every draw
    codes = (x / s.view(2, 1, 1, 1)).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, np.asarray(scales, np.float32)


def extend_q(seed, T, Hq, D, device):
    """Seeded bf16 queries [T, Hq, D] of an extend chunk."""
    import torch
    gen = torch.Generator(device=device).manual_seed(5_000_011 * (seed + 1) + T)
    return torch.randn((T, Hq, D), generator=gen, device=device).to(torch.bfloat16)


def global_scale_from_amax(amax):
    """The per-layer FP32 global scale used by the workloads: the layer's
    absolute maximum mapped onto E2M1 max x E4M3 max, amax / (6 * 448)."""
    a = np.float32(amax)
    return np.float32(a / np.float32(E2M1_MAX * E4M3_MAX)) if a > 0 else np.float32(1.0)


def fp8_scale_from_amax(amax):
    """FP8 per-tensor decode scale that maps the layer amax to the E4M3 maximum:
    amax / 448 in float32 (inputs recipe of the FP8 comparison workloads)."""
    return np.float32(np.float32(amax) / np.float32(448.0))


def slots_for(table_row, page_size, positions):
    pos = np.asarray(positions, dtype=np.int64)
    return np.asarray(table_row, np.int64)[pos // page_size] * page_size + pos % page_size


# --- the five workloads -------------------------------------------------------
TINY = Workload("tiny_nvfp4_d64", "nvfp4", 1, 2, 64, 1, 16, 256, 256,
                outliers=2, outlier_scale=8.0, outlier_kv="k", seed=0,
                notes="1 layer, 1 KV head, 2 query heads, D 64, one 256-token request, 16-token pages")
CTX32K = Workload("nvfp4_32k", "nvfp4", 4, 24, 256, 16, 64, 24576, 32768,
                  outliers=4, outlier_scale=10.0, seed=2, num_splits=0,
                  notes="27B-shaped full-attention layer, B16, lengths U[24K,32K], 64-token pages")
CTX160K = Workload("nvfp4_160k", "nvfp4", 4, 24, 256, 4, 64, 153600, 163840,
                   outliers=4, outlier_scale=10.0, seed=3, prefix_chunk=8192,
                   notes="B4, lengths U[150K,160K], plus an 8K-chunk prefix dequant of request 0")
CTX1M = Workload("nvfp4_1m", "nvfp4", 4, 24, 256, 1, 256, 1 << 20, 1 << 20,
                 dist="student_t4", seed=4, num_splits=128,
                 notes="B1 at 1,048,576 tokens, 256-token pages, 128 splits, Student-t(4) values")
INT4_220K = Workload("int4_220k", "int4", 2, 16, 256, 8, 1600, 220000, 220000, seed=5,
                     notes="INT4 per-token-head, 2 KV heads, 16 query heads, B8 at 220,000 tokens, 1600-token pages")

FP8_32K = Workload("fp8_32k", "fp8", 4, 24, 256, 16, 64, 24576, 32768,
                   outliers=4, outlier_scale=10.0, seed=2, num_splits=0,
                   notes="the 32K workload in the FP8 E4M3 per-tensor format (the comparison "
                         "the 4-bit cache is measured against)")

ALL = {w.name: w for w in (TINY, CTX32K, CTX160K, CTX1M, INT4_220K, FP8_32K)}
