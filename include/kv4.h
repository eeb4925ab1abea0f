/*
 * kv4.h -- C ABI of libkv4: a 4-bit paged KV cache for LLM decode on GB300
 * (sm_103a).
 *
 * The operations follow the three attention paths over one pool drawn in
 * Figure 2 of "SGLang's 4-bit KV cache: the 56% is exact, the 1.78x is
 * untested":
 *
 *   kv4_write             quantise new K/V tokens into the paged pool (the
 *                         pool holds packed E2M1 K and V, one E4M3 block
 *                         scale per 16 elements and FP32 global scales per
 *                         layer);
 *   kv4_decode_attention  decode attention that reads the 4-bit pool and
 *                         dequantises inside the kernel (decode is the only
 *                         path that reads the 4-bit cache directly), split
 *                         over the sequence with a log-sum-exp combine;
 *   kv4_dequant_prefix    the chunked-prefill path, first step: dequantise
 *                         the 4-bit prefix into an FP8 buffer that is reused;
 *   kv4_extend_attention  the chunked-prefill path, second step: the chunk's
 *                         queries attend over that FP8 prefix plus the FP8
 *                         current chunk, on the tensor cores;
 *   kv4_calibrate_global_scale  the per-layer FP32 global scales from the
 *                         layer's K and V at serving time;
 *   kv4_k8v4_write / kv4_k8v4_decode_attention  the k8v4 variant the same
 *                         page contrasts (FP8 keys, 4-bit values, both given
 *                         one fixed Hadamard rotation), KV4_K8V4 pools only.
 *
 * Three formats share the pool structure:
 *   KV4_NVFP4     E2M1 elements, one E4M3 scale per 16 elements, one FP32
 *                 global scale per layer for K and one for V; 9 bytes per 16
 *                 values, 0.5625 of FP8 (same page, "The 56% survives its own
 *                 scale").
 *   KV4_INT4_PTH  INT4 per token and head: 4-bit codes plus per-token-head
 *                 scales; at head_dim 256 each head of each token takes 264
 *                 bytes ("KV cache in 4 bits", section "What we changed").
 *   KV4_FP8       FP8 E4M3 with one FP32 scale per layer for K and one for V
 *                 (per tensor), 16 bytes per 16 values: the format the 4-bit
 *                 cache is compared against ("The 56% survives its own
 *                 scale").  Write and decode only.
 *
 * Encoding (the pages name the formats, not the encoder; this is the
 * library's definition, identical to the test oracle's):
 *   NVFP4, per 16-element block of a bf16 row x with global scale g (FP32):
 *     amax = max|x_i|; sf = amax / (6*g) [6*g rounded first]; S = E4M3(sf)
 *     with round-to-nearest-even, saturating at 448; denom = float(S) * g;
 *     if S == 0 or denom == 0 every code is +0, else
 *     code_i = E2M1(x_i / denom), RNE, saturating at 6, sign kept.
 *     All arithmetic is IEEE FP32.  Decode: e2m1(code) * e4m3(S) * g.
 *   INT4_PTH, per (token, head) row, separately for K and V:
 *     s = amax / 7 (FP32); code = clamp(rne(x / s), -8, 7); s == 0 gives
 *     all-zero codes.  Decode: code * s.
 *   FP8, per element with the layer's scale s: code = E4M3(x / s) (FP32
 *     quotient, RNE, saturating at 448, sign kept).  Decode: e4m3(code) * s.
 *   Two 4-bit codes per byte: element 2j in the low nibble of byte j.
 *
 * Pool layout (one pool per layer, caller-owned device memory):
 *   base -> [num_pages][num_kv_heads][chunk_bytes]; each (page, head) chunk
 *   holds these regions (P = page_size, D = head_dim):
 *     NVFP4: [K codes P*D/2][V codes P*D/2][K scales P*D/16][V scales P*D/16]
 *     INT4 : [K codes P*D/2][V codes P*D/2][K scale f32 * P][V scale f32 * P]
 *     FP8  : [K codes P*D]  [V codes P*D]
 *   chunk_bytes = P*(D + D/8) (NVFP4), P*(D + 8) (INT4), P*2*D (FP8).
 *   Row `off` of a region belongs to token `off` of the page, except the V
 *   codes of NVFP4 and INT4, stored in token pairs.  NVFP4: byte d of pair
 *   row p (D bytes) holds element d of token 2p in its low nibble and of
 *   token 2p+1 in its high nibble, and the pair's scale row (D/8 bytes)
 *   holds block b's scale of token 2p+i at byte 2b+i.  INT4: 32-bit word k
 *   of pair row p (D bytes) holds elements 4k .. 4k+3 of token 2p in its low
 *   16 bits and of token 2p+1 in its high 16 bits (element 4k+i in nibble i
 *   of the half); INT4 V scales stay one FP32 per token.  A slot is
 *   page * P + off.  The FP32 scales are not in the pool:
 *   callers pass them as a device float[2] = {g_K, g_V} per layer.
 *
 * Conventions for every entry point:
 *   - All device pointers are caller-owned; the library allocates nothing.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and never synchronises the host.
 *   - Arguments are validated on the host first.  A failure returns a status
 *     (and a message, kv4_last_error_message) and launches nothing.
 *   - Device-side range checks (a block_table entry outside [0, num_pages),
 *     a slot beyond the pool, seq_len beyond max_pages*P, a wait that ran
 *     out of time) never trap: the kernel skips the bad access, records a
 *     kv4_status in a per-device error word and returns normally.  Read and
 *     clear it with kv4_device_error().
 *   - Supported shapes: head_dim in {64, 128, 256}; page_size a positive
 *     multiple of 16; base 256-byte aligned; q, out and k/v 16-byte aligned.
 *   - Sizes are element counts unless named *_bytes.
 */
#ifndef KV4_H_
#define KV4_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { KV4_NVFP4 = 0, KV4_INT4_PTH = 1, KV4_FP8 = 2, KV4_K8V4 = 3 } kv4_fmt;

typedef enum {
  KV4_OK = 0,
  KV4_EINVAL = 1,        /* bad argument (null pointer, size, alignment)    */
  KV4_EUNSUPPORTED = 2,  /* valid but not built (e.g. head_dim 96)          */
  KV4_ECUDA = 3,         /* a CUDA runtime call or launch failed            */
  KV4_EBOUNDS = 4,       /* device: an index fell outside the pool/table    */
  KV4_ETIMEOUT = 5       /* device: a bounded wait on a copy ran out        */
} kv4_status;

/* One layer's paged pool.  Host-side descriptor; `base` is device memory of
 * kv4_pool_bytes() bytes. */
typedef struct {
  int32_t fmt;           /* kv4_fmt                                          */
  int32_t num_pages;
  int32_t page_size;     /* tokens per page (P)                              */
  int32_t num_kv_heads;  /* Hkv                                              */
  int32_t head_dim;      /* D                                                */
  int32_t reserved;      /* must be 0                                        */
  void*   base;
} kv4_pool;

/* Bytes of one (page, kv head) chunk and of the whole pool; 0 if the
 * descriptor is invalid.  Pure host functions. */
int64_t kv4_pool_chunk_bytes(const kv4_pool* pool);
int64_t kv4_pool_bytes(const kv4_pool* pool);

/*
 * kv4_write -- quantise T tokens of K and V into the pool (Figure 2: the
 * decode step stores the new token's K/V; prefill stores the prompt).
 *   k, v          device bf16 [T][Hkv][D], contiguous, 16-byte aligned.
 *   slot_mapping  device int64 [T]: destination slot of token t, or < 0 to
 *                 skip it.  A slot >= num_pages*P is skipped and flagged
 *                 KV4_EBOUNDS in the device error word.
 *   layer_global_scale  device float[2] {g_K, g_V}, each > 0: the NVFP4
 *                 global scales or the FP8 per-tensor scales (may be NULL for
 *                 INT4).
 *   fmt           must equal pool->fmt.
 * Writes only the rows of the slots it stores; nothing else in the pool.
 * Two tokens mapped to one slot race (last writer unspecified).
 */
kv4_status kv4_write(const void* k, const void* v, const int64_t* slot_mapping,
                     int64_t num_tokens, const kv4_pool* pool,
                     const float* layer_global_scale, int32_t fmt, void* stream);

/*
 * kv4_write_fp8 -- kv4_write fed with FP8 K/V, the form in which the engine
 * of Figure 2 ("SGLang's 4-bit KV cache") hands prompt and new-token K/V to
 * the cache.  k, v are device uint8 E4M3 codes [T][Hkv][D] (16-byte
 * aligned) with per-tensor scales in_scale = device float[2] {s_K, s_V};
 * each element is x = e4m3(code) * s as one IEEE FP32 product (round to
 * nearest), then encoded exactly as kv4_write encodes its bf16 values.
 * Other arguments, sizes and errors as kv4_write.
 */
kv4_status kv4_write_fp8(const void* k, const void* v, const float* in_scale,
                         const int64_t* slot_mapping, int64_t num_tokens, const kv4_pool* pool,
                         const float* layer_global_scale, int32_t fmt, void* stream);

/* Workspace bytes kv4_decode_attention needs for these sizes and this
 * num_splits (0 when num_splits == 1, which writes `out` directly).  Depends
 * on the current device's SM count. */
int64_t kv4_decode_workspace_bytes(int32_t batch, int32_t num_q_heads,
                                   int32_t head_dim, int32_t num_splits);

/*
 * kv4_decode_attention -- one decode step of paged attention over the 4-bit
 * pool (Figure 2: decode consumes the stored 4-bit codes and block scales
 * directly).  For request b and query head j (kv head
 * h = j / (Hq/Hkv): GQA groups are contiguous), over tokens t < seq_lens[b]
 * stored at slot block_table[b*max_pages + t/P]*P + t%P:
 *     out[b][j] = sum_t softmax_t(sm_scale * <q[b][j], K_hat_t>) V_hat_t
 * with K_hat/V_hat the decoded cache values.  seq_lens[b] == 0 gives a zero
 * row.  Work is cut along the sequence and the partial softmax states
 * (max, sum, weighted V) of the pieces are merged by a log-sum-exp combine:
 *   num_splits == 0  one wave of CTAs, each streaming an equal share of all
 *                    requests' tiles (balanced whatever the length mix);
 *   num_splits == 1  one CTA per (request, kv head, <= 8 query heads), which
 *                    writes `out` directly (no workspace, no combine);
 *   num_splits == S  as 0, and every request's range is also cut into S equal
 *                    splits, so each head's output merges at least S pieces.
 *   q            device bf16 [B][Hq][D]
 *   layer_global_scale  device float[2] {g_K, g_V} (NVFP4, FP8; NULL for INT4)
 *   block_table  device int32 [B][max_pages]; entries past a request's last
 *                page are never read.
 *   seq_lens     device int32 [B]; the decode step's own token (written by
 *                kv4_write beforehand) is included.
 *   num_splits   0..1024, see above.
 *   workspace    device scratch of >= kv4_decode_workspace_bytes() bytes
 *                (may be NULL when that is 0); contents on entry ignored.
 *   out          device [B][Hq][D], float32 if out_is_fp32 else bf16.
 * Deterministic: the same inputs give bitwise the same output.
 */
kv4_status kv4_decode_attention(const void* q, const kv4_pool* pool,
                                const float* layer_global_scale,
                                const int32_t* block_table, int32_t max_pages,
                                const int32_t* seq_lens, int32_t batch,
                                int32_t num_q_heads, float sm_scale,
                                int32_t num_splits, void* workspace,
                                int64_t workspace_bytes, void* out,
                                int32_t out_is_fp32, void* stream);

/*
 * kv4_decode_step -- one decode step with the step's new token written in
 * the same kernel: the effect of
 *     kv4_write(k_new, v_new, slot_mapping = the slot of position
 *               seq_lens[b] - 1 of each request b, T = B, ...)
 * followed by kv4_decode_attention(...) with the same arguments (Figure 2:
 * each decode step writes its token into the 4-bit cache and attends over
 * the request's tokens).  The new token's slot is the one the block table
 * gives position seq_lens[b] - 1 (no slot mapping is passed); a request with
 * seq_lens[b] == 0 writes nothing.  The CTA that decodes that position
 * quantises the token first, so the pool bytes written and the output are
 * bitwise those of the two calls.
 *   k_new, v_new  device bf16 [B][Hkv][D], 16-byte aligned.
 *   Other arguments as kv4_decode_attention.
 * NVFP4 and INT4 pools with at most 8 query heads per kv head; anything else
 * (FP8, k8v4, larger GQA groups) is KV4_EUNSUPPORTED: use the two calls.
 */
kv4_status kv4_decode_step(const void* q, const void* k_new, const void* v_new, const kv4_pool* pool,
                           const float* layer_global_scale, const int32_t* block_table,
                           int32_t max_pages, const int32_t* seq_lens, int32_t batch,
                           int32_t num_q_heads, float sm_scale, int32_t num_splits,
                           void* workspace, int64_t workspace_bytes, void* out,
                           int32_t out_is_fp32, void* stream);

/*
 * kv4_dequant_prefix -- the chunked-prefill path of Figure 2: the 4-bit
 * cached prefix is turned into FP8, in a buffer that is reused.  For each
 * request b, prefix token t < prefix_lens[b] and kv head h:
 *     ws[cu_prefix[b] + t][h][d] = E4M3(x_hat / s)
 * x_hat the FP32 decoded value ((e2m1*e4m3)*g for NVFP4, code*s for INT4),
 * s = fp8_scale[0] for K and fp8_scale[1] for V (per-tensor FP8 scales, the
 * consumer multiplies by s), FP32 division, E4M3 RNE saturating at 448.
 *   prefix_lens  device int32 [B]; cu_prefix device int64 [B+1] (exclusive
 *                prefix sums; rows of request b start at cu_prefix[b]).
 *   max_prefix_len  host upper bound of every prefix_lens[b] (sizes the
 *                grid); larger device values are clipped and flagged.
 *   fp8_scale    device float[2] {s_K, s_V}, each > 0.
 *   fp8_k, fp8_v device uint8 E4M3 [sum prefix_lens][Hkv][D].
 * A KV4_FP8 pool is already FP8: KV4_EUNSUPPORTED.
 */
kv4_status kv4_dequant_prefix(const kv4_pool* pool,
                              const float* layer_global_scale,
                              const int32_t* block_table, int32_t max_pages,
                              const int32_t* prefix_lens,
                              const int64_t* cu_prefix, int32_t batch,
                              int32_t max_prefix_len, const float* fp8_scale,
                              void* fp8_k, void* fp8_v, void* stream);

/*
 * kv4_extend_attention -- the chunked-prefill / extend attention of Figure 2
 * ("SGLang's 4-bit KV cache", right-hand column): the current chunk's
 * queries attend over the cached prefix (the FP8 workspace that
 * kv4_dequant_prefix wrote) plus the current chunk, which arrives as FP8
 * K/V.  For request b with prefix length Lp = prefix_lens[b] and chunk
 * length C = chunk_lens[b], chunk query i sits at position Lp + i and sees
 * every prefix key and chunk keys 0..i:
 *     out[i][j] = sum_k softmax_k(sm_scale * <q_ij, K_k>) V_k
 * over those keys of kv head j / (Hq / Hkv), K_k = e4m3(code) * fp8_scale[0],
 * V_k = e4m3(code) * fp8_scale[1] (one per-tensor scale pair for prefix and
 * chunk).  Computed on the tensor cores with f16 operands (exact for the FP8
 * values; q rounded to f16, |q| <= 65504 else KV4_EINVAL in the error word),
 * softmax weights rounded to f16 and FP32 accumulation.
 *   q            device bf16 [sum C][Hq][D]; row cu_chunk[b] + i is chunk
 *                token i of request b.
 *   chunk_k/v    device uint8 E4M3 [sum C][Hkv][D], same rows as q.
 *   prefix_k/v   device uint8 E4M3 [sum Lp][Hkv][D]; rows of request b start
 *                at cu_prefix[b] (the kv4_dequant_prefix layout).
 *   fp8_scale    device float[2] {s_K, s_V}, each > 0.
 *   prefix_lens, chunk_lens  device int32 [B] (>= 0, Lp + C < 2^31);
 *   cu_prefix, cu_chunk      device int64 [B+1] exclusive prefix sums.
 *   max_chunk_len  host upper bound of every chunk_lens[b] (sizes the grid);
 *                larger device values leave rows uncomputed and are flagged
 *                (KV4_EBOUNDS in the error word).
 *   sm_scale     > 0.   out  device [sum C][Hq][D], bf16 or FP32.
 *   workspace    NULL, or device scratch (256-byte aligned) of at least
 *                kv4_extend_workspace_bytes(B, max_chunk_len, Hq, D) bytes:
 *                the work is one CTA per (request, 128-row query tile,
 *                query head), one CTA per SM; with a workspace the items
 *                past the last full wave have their key ranges cut into
 *                pieces that fill one wave, and a second kernel merges the
 *                pieces' softmax states in a fixed order.  The result is the
 *                same function either way (up to FP32 summation order).
 * All device buffers 16-byte aligned (the int64 arrays 8-byte); Hq a
 * multiple of Hkv; head_dim 64, 128 or 256.  Asynchronous on `stream`;
 * allocates nothing.
 */
int64_t kv4_extend_workspace_bytes(int32_t batch, int32_t max_chunk_len, int32_t num_q_heads,
                                   int32_t head_dim);
kv4_status kv4_extend_attention(const void* q, const void* chunk_k, const void* chunk_v,
                                const void* prefix_k, const void* prefix_v,
                                const float* fp8_scale, const int32_t* prefix_lens,
                                const int64_t* cu_prefix, const int32_t* chunk_lens,
                                const int64_t* cu_chunk, int32_t batch, int32_t max_chunk_len,
                                int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                float sm_scale, void* workspace, int64_t workspace_bytes, void* out,
                                int32_t out_is_fp32, void* stream);

/*
 * kv4_calibrate_global_scale -- the NVFP4 global scales of one layer from its
 * K and V at serving time ("SGLang's 4-bit KV cache": Figure 2 keeps
 * per-layer FP32 global scales; the measured runs went without them, and
 * calibrating them is named as unfinished work).  For each of K and V:
 *     g = float32(amax) / 2688   (E2M1 max 6 x E4M3 max 448, FP32 rounding)
 * with amax the largest |x| over the tensor, and g = 1 when amax is not
 * positive.  The layer maximum then encodes to E4M3 scale 448 and code 6.
 *   k, v          device bf16 [T][Hkv][D], 16-byte aligned (T may be 0).
 *   layer_global_scale  device float[2], 8-byte aligned: receives {g_K, g_V}
 *                 (used as scratch while the maxima are reduced).
 * Inputs must be finite (a NaN gives g = 1).  Deterministic.
 */
kv4_status kv4_calibrate_global_scale(const void* k, const void* v, int64_t num_tokens,
                                      int32_t num_kv_heads, int32_t head_dim,
                                      float* layer_global_scale, void* stream);

/*
 * kv4_decode_attention_static_ws -- kv4_decode_attention for callers that
 * cannot allocate device memory.  The pages have no counterpart of this call;
 * it exists for library users, not for the method.
 *
 * Some callers cannot call cudaMalloc: code hosted by a framework that owns
 * every device allocation (for example an inference-server plugin held to a
 * fixed memory budget), or a decode loop that cannot take the device-wide
 * synchronisation an allocation may cause.  They pass the same inputs and
 * output as to kv4_decode_attention, without a workspace: the split partials
 * go to a scratch array inside the library instead.
 *   - The scratch is a fixed 8 MiB (8,388,608-byte) device array that every GPU
 *     loading the library holds until the process exits.  A call whose
 *     kv4_decode_workspace_bytes(batch, num_q_heads, head_dim, splits) exceeds
 *     it returns KV4_EINVAL (kv4_last_error_message gives both sizes) and
 *     launches nothing.  num_splits == 1 needs no scratch at all.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and keeps it; make that
 *     first call before any stream capture.  The kept address belongs to the
 *     device's context of that moment: cudaDeviceReset discards it together
 *     with the rest of the library's device state, so a process that resets a
 *     device must not call into the library on that device again.
 *   - Invalid arguments get the same status and message as from
 *     kv4_decode_attention; the scratch size is checked after them.
 *   - All calls share the one array and it keeps the last call's contents.
 *     Nothing in it needs to start at zero (each call writes every partial
 *     before reading it), but calls whose kernels overlap on the GPU -- on two
 *     streams, or from two host threads -- race on it: serialise them.
 *   - It allocates and frees nothing.  Results are bitwise those of
 *     kv4_decode_attention with the same num_splits.
 */
kv4_status kv4_decode_attention_static_ws(const void* q, const kv4_pool* pool,
                                          const float* layer_global_scale,
                                          const int32_t* block_table, int32_t max_pages,
                                          const int32_t* seq_lens, int32_t batch,
                                          int32_t num_q_heads, float sm_scale,
                                          int32_t num_splits, void* out,
                                          int32_t out_is_fp32, void* stream);

/*
 * The k8v4 variant ("SGLang's 4-bit KV cache", section "Against what this
 * site already established": the other 4-bit KV cache of the month stores
 * keys in FP8 and values in 4 bits and rotates both by one fixed FP32
 * Hadamard transform of size D).  KV4_K8V4 pools; chunk of P tokens =
 * [K codes P*D][V codes P*D/2][V scales FP32 * P]: K codes and V scales
 * in rows per token, V codes in token-pair rows by 16-bit halves as in the
 * INT4 pool.
 * Rotation H = S_D / sqrt(D) (Sylvester; symmetric, H H = I), evaluated on
 * the write path in FP32 as the fast Walsh-Hadamard transform (stages
 * len = 1, 2, ..., D/2, pairs (x_i, x_{i+len}) with bit len of i clear ->
 * (x_i + x_{i+len}, x_i - x_{i+len}), then times float32(1/sqrt(D))).
 * Keys: E4M3(k_rot / s_K), s_K = *key_scale (one FP32 scale per layer);
 * values: INT4 per (token, head), s = amax(v_rot) / 7,
 * code = clamp(rne(v_rot / s), -8, 7).  (The page names no value encoder;
 * this is the library's reading.)
 *
 * kv4_k8v4_write -- rotate and quantise T tokens of bf16 K/V
 *   ([T][Hkv][D], 16-byte aligned) into the pool at slot_mapping (int64
 *   [T], 8-byte aligned; < 0 skipped; beyond the pool flagged KV4_EBOUNDS).
 *   T * Hkv must be below 2^31 (else KV4_EINVAL).
 *
 * kv4_k8v4_decode_attention -- one decode step: q_rot = H q (bf16 q
 *   [B][Hq][D]), softmax(sm_scale * q_rot . K_hat_rot) over the request's
 *   tokens (block_table / seq_lens / max_pages as kv4_decode_attention),
 *   o = H (sum_t p_t V_hat_rot_t), out [B][Hq][D] bf16 or FP32.  The
 *   tiles of all (request, kv head) units are spread over one wave of
 *   persistent CTAs as in kv4_decode_attention, num_chunks (>= 1) being the
 *   number of split ranges per unit (num_splits there); the partial results
 *   always go through the workspace, and a second kernel merges them and
 *   applies H.  Workspace (256-byte aligned) of at least
 *   kv4_k8v4_workspace_bytes(B, Hkv, D, num_chunks) bytes (it depends on the
 *   device's SM count).  At most 8 query heads per kv head (else
 *   KV4_EUNSUPPORTED).  An empty request gives a zero row.  Asynchronous on
 *   `stream`; allocates nothing.
 */
kv4_status kv4_k8v4_write(const void* k, const void* v, const int64_t* slot_mapping,
                          int64_t num_tokens, const kv4_pool* pool, const float* key_scale,
                          void* stream);
int64_t kv4_k8v4_workspace_bytes(int32_t batch, int32_t num_kv_heads, int32_t head_dim,
                                 int32_t num_chunks);
kv4_status kv4_k8v4_decode_attention(const void* q, const kv4_pool* pool, const float* key_scale,
                                     const int32_t* block_table, int32_t max_pages,
                                     const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                                     float sm_scale, int32_t num_chunks, void* workspace,
                                     int64_t workspace_bytes, void* out, int32_t out_is_fp32,
                                     void* stream);

/* Read and clear the current device's error word (the first kv4_status a
 * kernel recorded since the last call, KV4_OK if none).  Synchronises the
 * device.  Returns KV4_ECUDA if the read itself fails. */
int32_t kv4_device_error(void);

/* Static text for a status code. */
const char* kv4_status_str(int32_t status);

/* Detail of the last host-side failure on the calling thread ("" if none). */
const char* kv4_last_error_message(void);

#ifdef __cplusplus
}
#endif

#endif /* KV4_H_ */
