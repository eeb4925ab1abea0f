"""Paged KV pool: request -> token -> slot -> bytes.

Test infrastructure only (see ``oracle/__init__.py``).

Figure 2 of "SGLang's 4-bit KV cache" shows one GPU KV pool holding packed
E2M1 K and V, the E4M3 block scales and per-layer FP32 global scales, with a
memory system that "maps request to token to slot".  "KV cache in 4 bits"
(section "What we changed") sizes an INT4 page as 211,200 bytes at 800 tokens
and 422,400 bytes at 1600 tokens, i.e. page_size * 264 bytes per KV head.

Layout (a reading; the pages do not fix byte order).  One pool per layer is a
byte array ``[num_pages][num_kv_heads][chunk_bytes]``; each (page, head)
chunk holds four regions, each a whole number of 16-byte units:

    NVFP4: [K codes P*D/2][V codes P*D/2][K scales P*D/16][V scales P*D/16]
    INT4 : [K codes P*D/2][V codes P*D/2][K scale f32 * P][V scale f32 * P]

so chunk_bytes = P*(D + D/8) for NVFP4 and P*(D + 8) for INT4.  Token
``off`` of a page owns row ``off`` of every region.  A slot is
``page * P + off``; a negative slot means "do not store".

The FP32 global scales are not in the pool array: they are passed beside it
as a float32 pair (K, V), as the caller owns them per layer.
"""
from dataclasses import dataclass

import numpy as np

from . import quant

NVFP4 = "nvfp4"
INT4 = "int4"


@dataclass(frozen=True)
class PoolSpec:
    fmt: str
    num_pages: int
    page_size: int
    num_kv_heads: int
    head_dim: int

    @property
    def code_bytes(self):            # packed 4-bit codes of one row
        return self.head_dim // 2

    @property
    def scale_bytes(self):           # scale bytes of one row (K or V)
        return self.head_dim // 16 if self.fmt == NVFP4 else 4

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
    """[N, row_bytes] byte indices of the rows (page, off) of one region."""
    width = spec.code_bytes if which in ("kc", "vc") else spec.scale_bytes
    base = spec.chunk_offset(page, head) + spec.region(which) + np.asarray(off, np.int64) * width
    return base[:, None] + np.arange(width, dtype=np.int64)[None, :]


def quantize_rows(spec, x_bf16, g):
    """Rows [..., D] of bf16 bits -> (codes bytes, scale bytes) in pool form."""
    if spec.fmt == NVFP4:
        return quant.nvfp4_quantize(x_bf16, g)
    codes, s = quant.int4_quantize(x_bf16)
    return codes, s.astype(np.float32).view(np.uint8).reshape(s.shape + (4,))


def write(pool, spec, k, v, slot_mapping, gscale):
    """Store tokens into the pool (the write path of Figure 2).

    k, v: uint16 bf16 bits [T, Hkv, D]; slot_mapping: int64 [T]; gscale:
    float32 [2] = (g_K, g_V), used by NVFP4 only.  Slots < 0 are skipped.
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
            pool[_row_index(spec, page, off, h, name + "c")] = codes[:, h]
            pool[_row_index(spec, page, off, h, name + "s")] = scales[:, h].reshape(len(keep), -1)
    return pool


def token_pages(block_table_row, positions, page_size):
    """Logical token positions of one request -> (physical page, offset)."""
    pos = np.asarray(positions, dtype=np.int64)
    return np.asarray(block_table_row, dtype=np.int64)[pos // page_size], pos % page_size


def read_rows(pool, spec, page, off, head, gscale, kind):
    """Dequantised float64 rows [N, D] of K (kind='k') or V (kind='v')."""
    codes = pool[_row_index(spec, page, off, head, kind + "c")]
    sbytes = pool[_row_index(spec, page, off, head, kind + "s")]
    if spec.fmt == NVFP4:
        g = gscale[0] if kind == "k" else gscale[1]
        return quant.nvfp4_dequantize(codes, sbytes, g)
    s = np.ascontiguousarray(sbytes).view(np.float32).reshape(-1)
    return quant.int4_dequantize(codes, s)
