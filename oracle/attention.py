"""Exact attention over the dequantised 4-bit cache, the split-KV combine,
and the dequantisation of a cached prefix into an FP8 workspace.

Test infrastructure only (see ``oracle/__init__.py``).

Figure 2 of "SGLang's 4-bit KV cache" has three paths over one pool: decode
alone reads the 4-bit codes, dequantising them in the kernel; chunked
prefill / extend first turns the cached prefix into FP8, in a buffer that is
reused, then attends over that prefix plus the chunk.  The decode reference here is the plain definition:
for request b and query head j (GQA groups are contiguous, kv head
h = j // (Hq / Hkv)), over the request's tokens t < seq_len[b] at slot
block_table[b][t // P] * P + t % P,

    score_t = sm_scale * <q_j, K_hat_t>,   out_j = sum_t softmax(score)_t V_hat_t

in float64 with the maximum subtracted.  K_hat / V_hat are the decoded cache
values, so this measures kernel parity, not quantisation error.  A request
with seq_len 0 yields a zero row.

The split-KV log-sum-exp combine (a step the pages do not describe; it is how
one long request is spread over many cores) is restated in ``lse_combine``.
"""
import numpy as np

from . import pool as pool_mod
from .formats import bf16_to_f32, e2m1_decode, e4m3_decode, e4m3_encode
from .quant import _unpack_nibbles, NVFP4_BLOCK

_CHUNK = 1 << 16   # tokens dequantised at a time (memory bound only)


def _kv_rows(pool, spec, gscale, bt_row, h, lo, hi, kind):
    page, off = pool_mod.token_pages(bt_row, np.arange(lo, hi), spec.page_size)
    return pool_mod.read_rows(pool, spec, page, off, h, gscale, kind)


def decode_attention(q, pool, spec, gscale, block_table, seq_lens, sm_scale, rows=None):
    """FP64 decode attention.

    q: uint16 bf16 bits [B, Hq, D]; block_table int [B, max_pages];
    seq_lens int [B]; sm_scale float32.  ``rows``: optional list of (b, j)
    to compute (the rest stay NaN).  Returns float64 [B, Hq, D].
    """
    B, Hq, D = q.shape
    Hkv = spec.num_kv_heads
    assert Hq % Hkv == 0
    G = Hq // Hkv
    sm = np.float64(np.float32(sm_scale))
    out = np.full((B, Hq, D), np.nan if rows is not None else 0.0)
    want = {}
    for b, j in (rows if rows is not None else [(b, j) for b in range(B) for j in range(Hq)]):
        want.setdefault((b, j // G), []).append(j)
    for (b, h), js in sorted(want.items()):
        L = int(seq_lens[b])
        js = sorted(js)
        if L == 0:
            out[b, js] = 0.0
            continue
        Q = bf16_to_f32(q[b, js]).astype(np.float64)                  # [g, D]
        scores = np.empty((len(js), L))
        for lo in range(0, L, _CHUNK):
            hi = min(L, lo + _CHUNK)
            K = _kv_rows(pool, spec, gscale, block_table[b], h, lo, hi, "k")
            scores[:, lo:hi] = sm * (Q @ K.T)
        scores -= scores.max(axis=1, keepdims=True)
        p = np.exp(scores)
        acc = np.zeros((len(js), D))
        for lo in range(0, L, _CHUNK):
            hi = min(L, lo + _CHUNK)
            V = _kv_rows(pool, spec, gscale, block_table[b], h, lo, hi, "v")
            acc += p[:, lo:hi] @ V
        out[b, js] = acc / p.sum(axis=1, keepdims=True)
    return out


def split_partials(scores, values, bounds):
    """Per-split softmax partials over token ranges [bounds[i], bounds[i+1]).

    scores float64 [L], values float64 [L, D].  Returns (m [S], l [S],
    o [S, D]) with m the split maximum (-inf if empty), l = sum exp(s - m),
    o = sum exp(s - m) * v.
    """
    S = len(bounds) - 1
    m = np.full(S, -np.inf)
    l = np.zeros(S)
    o = np.zeros((S, values.shape[1]))
    for i in range(S):
        a, b = bounds[i], bounds[i + 1]
        if b > a:
            m[i] = scores[a:b].max()
            e = np.exp(scores[a:b] - m[i])
            l[i] = e.sum()
            o[i] = e @ values[a:b]
    return m, l, o


def lse_combine(m, l, o):
    """Merge split partials: m* = max m_s, w_s = exp(m_s - m*),
    out = sum w_s o_s / sum w_s l_s (zero if every split is empty)."""
    m = np.asarray(m, dtype=np.float64)
    if not np.any(np.isfinite(m)):
        return np.zeros(np.asarray(o).shape[1])
    mstar = m[np.isfinite(m)].max()
    w = np.where(np.isfinite(m), np.exp(np.where(np.isfinite(m), m, 0.0) - mstar), 0.0)
    return (w[:, None] * o).sum(axis=0) / (w * l).sum()


def _dequant_f32(pool, spec, gscale, page, off, h, kind):
    """Decoded rows in float32 as the prefix path computes them:
    NVFP4 (e2m1 * e4m3) * g, INT4 code * s -- each product rounded to float32."""
    codes = pool_mod.get_codes(pool, spec, page, off, h, kind)
    sb = pool_mod.get_scales(pool, spec, page, off, h, kind)
    n = _unpack_nibbles(codes)
    if spec.fmt == pool_mod.NVFP4:
        g = np.float32(gscale[0] if kind == "k" else gscale[1])
        e = e2m1_decode(n).astype(np.float32)
        s = e4m3_decode(sb).astype(np.float32)
        D = e.shape[-1]
        es = (e.reshape(e.shape[0], D // NVFP4_BLOCK, NVFP4_BLOCK) * s[:, :, None]).astype(np.float32)
        return (es.reshape(e.shape[0], D) * g).astype(np.float32)
    c = n.astype(np.int64)
    c = np.where(c >= 8, c - 16, c).astype(np.float32)
    s = np.ascontiguousarray(sb).view(np.float32).reshape(-1)
    return (c * s[:, None]).astype(np.float32)


def dequant_prefix(pool, spec, gscale, block_table, prefix_lens, fp8_scale):
    """Cached prefix -> FP8 E4M3 workspace (the chunked-prefill path).

    For every request b and prefix token t < prefix_lens[b], row
    cu[b] + t of the workspaces (cu = exclusive prefix sum of prefix_lens)
    holds, for each kv head, E4M3(x_hat / s) with s = fp8_scale[0] for K and
    fp8_scale[1] for V, x_hat the float32 decoded value, division in float32,
    E4M3 rounding RNE and saturating.  Returns (ws_k, ws_v) uint8
    [sum prefix_lens, Hkv, D].
    """
    Hkv, D = spec.num_kv_heads, spec.head_dim
    total = int(np.sum(prefix_lens))
    ws = {"k": np.zeros((total, Hkv, D), np.uint8), "v": np.zeros((total, Hkv, D), np.uint8)}
    row = 0
    for b, n in enumerate(prefix_lens):
        n = int(n)
        for lo in range(0, n, _CHUNK):
            hi = min(n, lo + _CHUNK)
            page, off = pool_mod.token_pages(block_table[b], np.arange(lo, hi), spec.page_size)
            for h in range(Hkv):
                for kind, s in (("k", np.float32(fp8_scale[0])), ("v", np.float32(fp8_scale[1]))):
                    xh = _dequant_f32(pool, spec, gscale, page, off, h, kind)
                    ws[kind][row + lo:row + hi, h] = e4m3_encode((xh / s).astype(np.float32))
        row += n
    return ws["k"], ws["v"]


def extend_attention(q, chunk_k, chunk_v, prefix_k, prefix_v, fp8_scale, prefix_lens,
                     chunk_lens, sm_scale, rows=None):
    """FP64 chunked-prefill / extend attention over an FP8 prefix plus an FP8 chunk.

    Figure 2 of "SGLang's 4-bit KV cache", right-hand column: the current
    chunk arrives as FP8 K/V, the cached prefix has been dequantised into the
    FP8 workspace (``dequant_prefix``), and the chunk's queries attend over
    prefix plus chunk.  For request b with prefix length Lp = prefix_lens[b]
    and chunk length C = chunk_lens[b], the key sequence is the Lp prefix rows
    followed by the C chunk rows; chunk query i sits at position Lp + i and
    sees keys 0 .. Lp + i (all of the prefix, and the chunk causally up to
    itself).  Values are e4m3(code) * s with s = fp8_scale[0] for K and
    fp8_scale[1] for V (one per-tensor scale pair for prefix and chunk), and

        out[i, j] = sum_k softmax_k(sm_scale * <q_ij, K_k>) V_k

    over the visible keys of kv head j // (Hq / Hkv), in float64.

    q: uint16 bf16 bits [sum C, Hq, D]; chunk_k/v: uint8 E4M3 [sum C, Hkv, D];
    prefix_k/v: uint8 E4M3 [sum Lp, Hkv, D]; rows of request b start at the
    exclusive prefix sums of chunk_lens / prefix_lens.  rows: optional
    iterable of (chunk row, query head) to compute; others stay zero.
    Returns float64 [sum C, Hq, D].
    """
    T, Hq, D = q.shape
    Hkv = chunk_k.shape[1]
    G = Hq // Hkv
    sk, sv = float(np.float32(fp8_scale[0])), float(np.float32(fp8_scale[1]))
    out = np.zeros((T, Hq, D), np.float64)
    cu_c = np.concatenate([[0], np.cumsum(np.asarray(chunk_lens, np.int64))])
    cu_p = np.concatenate([[0], np.cumsum(np.asarray(prefix_lens, np.int64))])
    want = None if rows is None else {}
    if rows is not None:
        for r, j in rows:
            want.setdefault(int(r), set()).add(int(j))
    for b in range(len(chunk_lens)):
        C, Lp = int(chunk_lens[b]), int(prefix_lens[b])
        if C == 0:
            continue
        r0, p0 = int(cu_c[b]), int(cu_p[b])
        sel = range(C) if want is None else sorted(i - r0 for i in want if r0 <= i < r0 + C)
        if not sel:
            continue
        for h in range(Hkv):
            keys = np.concatenate([e4m3_decode(prefix_k[p0:p0 + Lp, h]),
                                   e4m3_decode(chunk_k[r0:r0 + C, h])]) * sk
            vals = np.concatenate([e4m3_decode(prefix_v[p0:p0 + Lp, h]),
                                   e4m3_decode(chunk_v[r0:r0 + C, h])]) * sv
            for j in range(h * G, (h + 1) * G):
                for i in sel:
                    if want is not None and j not in want[r0 + i]:
                        continue
                    n = Lp + i + 1                      # visible keys of query i
                    qv = bf16_to_f32(q[r0 + i, j]).astype(np.float64)
                    s = float(sm_scale) * (keys[:n] @ qv)
                    p = np.exp(s - s.max())
                    out[r0 + i, j] = (p @ vals[:n]) / p.sum()
    return out
