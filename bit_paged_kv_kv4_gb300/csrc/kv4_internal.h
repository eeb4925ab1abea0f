// Internal interfaces between the C ABI (kv4_abi.cu) and the kernel files.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <nvtx3/nvToolsExt.h>

#include "../../include/kv4.h"

namespace kv4 {

// An NVTX range around one C-ABI call: named in Nsight timelines, and a
// no-op (the header-only NVTX v3 API) when no tool is attached.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// Division of n < 2^31 by a fixed d in [1, 2^31) with one multiply-high, an
// add and a shift (T. Granlund, P. Montgomery, "Division by invariant integers
// using multiplication", PLDI 1994, section 4): s = ceil(log2 d),
// m = floor(2^32 (2^s - d) / d) + 1, n / d = (mulhi(n, m) + n) >> s.
struct FastDiv {
  uint32_t d, m, s;
};
inline FastDiv make_fastdiv(uint32_t d) {
  uint32_t s = 0;
  while ((uint64_t{1} << s) < d) ++s;
  const uint64_t m = ((uint64_t{1} << 32) * ((uint64_t{1} << s) - d)) / d + 1;
  return FastDiv{d, static_cast<uint32_t>(m), s};
}


struct DecodeArgs {
  const uint8_t* pool;
  int64_t chunk_bytes;
  int P, Hkv, num_pages, D, fmt;
  const __nv_bfloat16* q;       // [B][Hq][D]
  const float* gscale;          // [2] (NVFP4) or null
  const int32_t* block_table;   // [B][max_pages]
  int max_pages;
  const int32_t* seq_lens;      // [B]
  int B, Hq, G;
  float sm_scale;
  int num_splits;               // split ranges per unit (>= 1)
  int n_cta;                    // CTAs launched
  int unit_ctas;                // 1: one CTA per unit, output written directly
  int box_rows;                 // rows per TMA box of the code-row map (16 or 32)
  int tile;                     // tokens per tile (decode_tile_tokens(fmt))
  int64_t* cum;                 // [B+1] tile offsets of each request (balanced mode)
  float* part_ml;               // [slots][8][4]: m_x, l, m_y, 0
  float* part_o;                // [slots][8][D]
  void* out;
  int out_f32;
  int* err;
  // kv4_decode_step: each request's new K/V token ([B][Hkv][D] bf16), written
  // into its position seq_lens[b] - 1 by the CTA that decodes that position;
  // null for a plain decode
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
};

struct WriteArgs {
  const __nv_bfloat16* k;       // [T][Hkv][D]
  const __nv_bfloat16* v;
  const int64_t* slot_mapping;  // [T]
  int64_t T;
  uint8_t* pool;
  int64_t chunk_bytes;
  int P, Hkv, num_pages, D, fmt;
  const float* gscale;
  int* err;
  int rows;                     // T * Hkv (< 2^31)
  FastDiv hkv_div, p_div;       // by Hkv, by P
  const uint8_t* k8;            // FP8-input write: E4M3 [T][Hkv][D] (else null)
  const uint8_t* v8;
  const float* in_scale;        // [2] {s_K, s_V} of the FP8 input
  uint32_t units;               // ceil(T / 2) * Hkv * D / 16 (token pair, head, 16-element block)
  int sms;                      // SMs of the device (sizes the grid)
};

struct PrefixArgs {
  const uint8_t* pool;
  int64_t chunk_bytes;
  int P, Hkv, num_pages, D, fmt;
  const float* gscale;
  const int32_t* block_table;
  int max_pages;
  const int32_t* prefix_lens;
  const int64_t* cu_prefix;
  int B, max_prefix_len;
  const float* fp8_scale;
  uint8_t* out_k;
  uint8_t* out_v;
  int* err;
  FastDiv hkv_div, p_div;       // by Hkv, by P
  int sms;                      // SMs of the device (sizes the grid)
};

// `map`: the code-row view (FP8) or the 3-D code view (NVFP4, INT4); `smap`:
// the 3-D scale view (NVFP4, INT4; ignored for FP8).
cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& map, const CUtensorMap& smap,
                          cudaStream_t st);
cudaError_t launch_write(const WriteArgs& a, cudaStream_t st);
// mk / mv: the K / V workspaces as 2-D byte tensors of 128-byte rows (boxes of
// 128 bytes x 16 rows, 128-byte swizzle) for the kernel's tensor stores.
cudaError_t launch_prefix(const PrefixArgs& a, const CUtensorMap& mk, const CUtensorMap& mv, cudaStream_t st);

struct CalibArgs {
  const __nv_bfloat16* k;       // [n] elements (T * Hkv * D)
  const __nv_bfloat16* v;
  int64_t n;
  float* out;                   // [2]
};
cudaError_t launch_calibrate(const CalibArgs& a, cudaStream_t st);

struct ExtendArgs {
  const __nv_bfloat16* q;       // [sum C][Hq][D]
  const uint8_t* ck;            // E4M3 [sum C][Hkv][D]
  const uint8_t* cv;
  const uint8_t* pk;            // E4M3 [sum Lp][Hkv][D]
  const uint8_t* pv;
  const float* fp8_scale;       // [2] {s_K, s_V}
  const int32_t* prefix_lens;   // [B]
  const int64_t* cu_prefix;     // [B+1]
  const int32_t* chunk_lens;    // [B]
  const int64_t* cu_chunk;      // [B+1]
  int B, max_chunk_len, Hq, Hkv, D, G;
  float sm_scale;
  void* out;                    // [sum C][Hq][D] bf16 or f32
  int out_f32;
  int* err;
  // Work list: items (request, 128-row query tile, query head), longest
  // first; the last `split` items are cut into `ways` key ranges whose
  // partial states go to part_o / part_ml and are merged by a second kernel.
  int qtiles;                   // query tiles per request: ceil(max_chunk_len / 128)
  int items;                    // B * qtiles * Hq
  int split, ways;
  float* part_o;                // [split * ways][128][D] unnormalised O
  float* part_ml;               // [split * ways][128][2] (base m in log2 units, l)
};
cudaError_t launch_extend(const ExtendArgs& a, cudaStream_t st);
// Split of the extend work list for `sms` SMs: the remainder items of the
// last partial wave are cut into ways pieces so they fill one wave.
void extend_split(int items, int sms, int& split, int& ways);

struct K8V4WriteArgs {
  const __nv_bfloat16* k;       // [T][Hkv][D]
  const __nv_bfloat16* v;
  const int64_t* slot_mapping;  // [T]
  int64_t rows;                 // T * Hkv
  uint8_t* pool;
  int64_t chunk_bytes;
  int P, Hkv, num_pages, D;
  const float* s_k;             // [1] FP8 key scale
  int* err;
  FastDiv hkv_div, p_div;       // by Hkv, by P (set by the launch)
};
cudaError_t launch_k8v4_write(const K8V4WriteArgs& a, cudaStream_t st);
int decode_tile_tokens(int fmt);
// Sets the message kv4_last_error_message() returns on this thread.
void set_error_message(const char* msg);
// Resident CTAs per SM of the decode kernel for `fmt`, and the largest over
// formats (the workspace is sized for it).
int decode_ctas_per_sm(int fmt);
int decode_max_ctas_per_sm();
// The NVFP4 / INT4 decode kernel (kv4_decode4.cu) and its resident CTAs per SM.
cudaError_t launch_decode4(const DecodeArgs& a, const CUtensorMap& cmap, const CUtensorMap& smap,
                           cudaStream_t st);
int decode4_ctas_per_sm();
// Every argument check of kv4_decode_attention except those of the workspace
// (the message goes to kv4_last_error_message); KV4_OK when all pass.
kv4_status check_decode_args(const void* q, const kv4_pool* pool, const float* layer_global_scale,
                             const int32_t* block_table, int32_t max_pages, const int32_t* seq_lens,
                             int32_t batch, int32_t num_q_heads, float sm_scale, int32_t num_splits,
                             const void* out);

}  // namespace kv4
