"""Paged KV pool: request -> token -> slot -> bytes.

Test infrastructure only (see ``oracle/__init__.py``).

Figure 2 of "SGLang's 4-bit KV cache" shows one GPU KV pool holding packed
E2M1 K and V, the E4M3 block scales and per-layer FP32 global scales, and a
memory system that takes each request's tokens to pool slots.  "KV cache in 4 bits"
(section "What we changed") sizes an INT4 page as 211,200 bytes at 800 tokens
and 422,400 bytes at 1600 tokens, i.e. page_size * 264 bytes per KV head.

Layout (a reading; the pages do not fix byte order).  One pool per layer is a
byte array ``[num_pages][num_kv_heads][chunk_bytes]``; each (page, head)
chunk holds four regions, each a whole number of 16-byte units:

    NVFP4: [K codes P*D/2][V codes P*D/2][K scales P*D/16][V scales P*D/16]
    INT4 : [K codes P*D/2][V codes P*D/2][K scale f32 * P][V scale f32 * P]
    FP8  : [K codes P*D]  [V codes P*D]   (per-tensor scales beside the pool)

so chunk_bytes = P*(D + D/8) for NVFP4, P*(D + 8) for INT4, P*2*D for FP8.

Row order inside a region:

* K codes and scales, INT4 V scales and every FP8 region: token ``off`` of
  the page owns row ``off`` (D/2 code bytes, element 2j in the low nibble
  of byte j; D/16 scale bytes, or one FP32 scale; FP8: D code bytes,
  element d in byte d).
* NVFP4 V: tokens are stored in pairs (2p, 2p+1).  Code byte d of pair row p
  (D bytes) holds element d of token 2p in its low nibble and element d of
  token 2p+1 in its high nibble; scale byte 2*blk + i of pair row p (D/8
  bytes) is block blk of token 2p+i.  A decode kernel contracts V over
  tokens, so its tensor-core operands pair two tokens of one element: this
  order hands it those pairs as they are stored.  Sizes are unchanged.
* INT4 V codes: also in token pairs, interleaved by 16-bit halves.  Pair
  row p (D bytes) is D/8 words of 4 bytes; word k holds elements 4k .. 4k+3
  of token 2p in its low half and of token 2p+1 in its high half (element
  4k+i in nibble i of the half).  Bytes 2k, 2k+1 of a token's packed row
  are bytes 4k + 2i, 4k + 2i + 1 of the pair row, i = off % 2.  A decode
  kernel's shift by 4 or 8 bits of such a word lines up one element of both
  tokens in the two halves of a 32-bit register, the form its INT4 -> f16
  conversion takes.

A slot is ``page * P + off``; a negative slot means "do not store".

The FP32 global scales are not in the pool array: they are passed beside it
as a float32 pair (K, V), as the caller owns them per layer.
"""
from dataclasses import dataclass

import numpy as np

from . import quant

NVFP4 = "nvfp4"
INT4 = "int4"
FP8 = "fp8"


@dataclass(frozen=True)
class PoolSpec:
    fmt: str
    num_pages: int
    page_size: int
    num_kv_heads: int
    head_dim: int

    @property
    def code_bytes(self):            # codes of one row: packed 4-bit, or one byte each (FP8)
        return self.head_dim if self.fmt == FP8 else self.head_dim // 2

    @property
    def scale_bytes(self):           # scale bytes of one row (K or V)
        return {NVFP4: self.head_dim // 16, INT4: 4, FP8: 0}[self.fmt]

    @property
    def chunk_bytes(self):           # one (page, kv head) chunk, K and V
        return self.page_size * 2 * (self.code_bytes + self.scale_bytes)

    @property
    def pool_bytes(self):
        return self.num_pages * self.num_kv_heads * self.chunk_bytes

    def region(self, which):
        """Byte offset of region 'kc', 'vc', 'ks' or 'vs' inside a chunk."""
        P = self.page_size
        return {"kc": 0, "vc": P * self.code_bytes,
                "ks": 2 * P * self.code_bytes,
                "vs": 2 * P * self.code_bytes + P * self.scale_bytes}[which]

    def chunk_offset(self, page, head):
        return (np.asarray(page, dtype=np.int64) * self.num_kv_heads + head) * self.chunk_bytes


def new_pool(spec, fill=0):
    return np.full(spec.pool_bytes, fill, dtype=np.uint8)


def _row_index(spec, page, off, head, which):
    """[N, row_bytes] byte indices of token rows (page, off) of a region stored
    one row per token (K codes and scales; every INT4 region)."""
    width = spec.code_bytes if which in ("kc", "vc") else spec.scale_bytes
    base = spec.chunk_offset(page, head) + spec.region(which) + np.asarray(off, np.int64) * width
    return base[:, None] + np.arange(width, dtype=np.int64)[None, :]


def _pair_v(spec):
    return spec.fmt == NVFP4


def _pair_v16(spec):
    return spec.fmt == INT4


def _v_pair16_codes_index(spec, page, off, head):
    """INT4 V codes: [N, D/2] byte indices of the packed bytes of tokens
    (page, off) inside their pair rows (byte 2k + j of the token's packed row
    at 4k + 2 (off % 2) + j of the pair row)."""
    off = np.asarray(off, np.int64)
    D = spec.head_dim
    j = np.arange(D // 2, dtype=np.int64)
    col = 4 * (j // 2) + (j % 2)
    base = spec.chunk_offset(page, head) + spec.region("vc") + (off // 2) * D + 2 * (off & 1)
    return base[:, None] + col[None, :]


def _v_pair_codes_index(spec, page, off, head):
    """NVFP4 V codes: [N, D] byte indices of the pair rows of tokens (page,
    off) and [N] nibble shifts (0 for even tokens, 4 for odd)."""
    off = np.asarray(off, np.int64)
    D = spec.head_dim
    base = spec.chunk_offset(page, head) + spec.region("vc") + (off // 2) * D
    return base[:, None] + np.arange(D, dtype=np.int64)[None, :], (off & 1) * 4


def _v_pair_scales_index(spec, page, off, head):
    """NVFP4 V scales: [N, D/16] byte indices of the scales of tokens (page, off)."""
    off = np.asarray(off, np.int64)
    W = spec.scale_bytes
    base = spec.chunk_offset(page, head) + spec.region("vs") + (off // 2) * (2 * W) + (off & 1)
    return base[:, None] + 2 * np.arange(W, dtype=np.int64)[None, :]


def get_codes(pool, spec, page, off, head, kind):
    """Packed codes [N, D/2] (element 2j in the low nibble of byte j) of tokens
    (page, off), whatever the region's row order."""
    if kind == "v" and _pair_v(spec):
        idx, sh = _v_pair_codes_index(spec, page, off, head)
        nib = (pool[idx] >> sh[:, None].astype(np.uint8)) & 0xF
        return (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    if kind == "v" and _pair_v16(spec):
        return pool[_v_pair16_codes_index(spec, page, off, head)]
    return pool[_row_index(spec, page, off, head, kind + "c")]


def get_scales(pool, spec, page, off, head, kind):
    """Scale bytes [N, row_scale_bytes] of tokens (page, off)."""
    if kind == "v" and _pair_v(spec):
        return pool[_v_pair_scales_index(spec, page, off, head)]
    return pool[_row_index(spec, page, off, head, kind + "s")]


def put_rows(pool, spec, page, off, head, kind, codes, scales):
    """Store packed codes [N, D/2] and scale bytes [N, W] of tokens (page, off),
    touching nothing else (for paired V rows, only the token's own nibbles)."""
    if kind == "v" and _pair_v(spec):
        idx, sh = _v_pair_codes_index(spec, page, off, head)
        c = np.asarray(codes, np.uint8)
        nib = np.empty((c.shape[0], 2 * c.shape[1]), np.uint8)
        nib[:, 0::2] = c & 0xF
        nib[:, 1::2] = c >> 4
        for r in range(idx.shape[0]):               # one token at a time: pairs may repeat
            s = int(sh[r])
            old = pool[idx[r]]
            pool[idx[r]] = (old & np.uint8(0xF0 >> s)) | (nib[r] << np.uint8(s))
        pool[_v_pair_scales_index(spec, page, off, head)] = scales
        return
    if kind == "v" and _pair_v16(spec):
        pool[_v_pair16_codes_index(spec, page, off, head)] = codes     # the token's own bytes only
        pool[_row_index(spec, page, off, head, "vs")] = scales
        return
    pool[_row_index(spec, page, off, head, kind + "c")] = codes
    pool[_row_index(spec, page, off, head, kind + "s")] = scales


def quantize_rows(spec, x_bf16, g):
    """Rows [..., D] of bf16 bits or float32 values -> (codes bytes, scale bytes) in pool form."""
    if spec.fmt == NVFP4:
        return quant.nvfp4_quantize(x_bf16, g)
    if spec.fmt == FP8:
        codes = quant.fp8_quantize(x_bf16, g)
        return codes, np.zeros(codes.shape[:-1] + (0,), np.uint8)
    codes, s = quant.int4_quantize(x_bf16)
    return codes, s.astype(np.float32).view(np.uint8).reshape(s.shape + (4,))


def write(pool, spec, k, v, slot_mapping, gscale):
    """Store tokens into the pool (the write path of Figure 2).

    k, v: uint16 bf16 bits (or float32 values) [T, Hkv, D]; slot_mapping: int64 [T]; gscale:
    float32 [2] = (g_K, g_V): NVFP4 global scales or FP8 per-tensor scales
    (unused for INT4).  Slots < 0 are skipped.
    """
    slot = np.asarray(slot_mapping, dtype=np.int64)
    keep = np.nonzero(slot >= 0)[0]
    if keep.size == 0:
        return pool
    assert np.all(slot[keep] < spec.num_pages * spec.page_size)
    page, off = slot[keep] // spec.page_size, slot[keep] % spec.page_size
    gk, gv = np.float32(gscale[0]), np.float32(gscale[1])
    for name, x, g in (("k", k, gk), ("v", v, gv)):
        codes, scales = quantize_rows(spec, np.asarray(x)[keep], g)
        for h in range(spec.num_kv_heads):
            put_rows(pool, spec, page, off, h, name, codes[:, h], scales[:, h].reshape(len(keep), -1))
    return pool


def write_fp8(pool, spec, k_codes, v_codes, in_scale, slot_mapping, gscale):
    """The write fed with FP8 K/V, as the engine hands them to the cache
    ("SGLang's 4-bit KV cache", Figure 2: prompt and new-token K/V arrive as
    FP8): k_codes, v_codes uint8 E4M3 [T, Hkv, D] with per-tensor scales
    in_scale = (s_K, s_V); each value is e4m3(code) * s as one float32
    product, then encoded exactly as ``write`` encodes its bf16 values."""
    k = quant.fp8_input_values(k_codes, np.float32(in_scale[0]))
    v = quant.fp8_input_values(v_codes, np.float32(in_scale[1]))
    return write(pool, spec, k, v, slot_mapping, gscale)


def token_pages(block_table_row, positions, page_size):
    """Logical token positions of one request -> (physical page, offset)."""
    pos = np.asarray(positions, dtype=np.int64)
    return np.asarray(block_table_row, dtype=np.int64)[pos // page_size], pos % page_size


def read_rows(pool, spec, page, off, head, gscale, kind):
    """Dequantised float64 rows [N, D] of K (kind='k') or V (kind='v')."""
    codes = get_codes(pool, spec, page, off, head, kind)
    sbytes = get_scales(pool, spec, page, off, head, kind)
    if spec.fmt == NVFP4:
        g = gscale[0] if kind == "k" else gscale[1]
        return quant.nvfp4_dequantize(codes, sbytes, g)
    if spec.fmt == FP8:
        return quant.fp8_dequantize(codes, gscale[0] if kind == "k" else gscale[1])
    s = np.ascontiguousarray(sbytes).view(np.float32).reshape(-1)
    return quant.int4_dequantize(codes, s)
