// Internal interfaces between the C ABI (kv4_abi.cu) and the kernel files.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace kv4 {

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
  int num_splits;
  float* part_ml;               // [B][Hq][S][4]: m_x, l, m_y, 0
  float* part_o;                // [B][Hq][S][D]
  void* out;
  int out_f32;
  int* err;
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
};

cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& map, cudaStream_t st);
cudaError_t launch_write(const WriteArgs& a, cudaStream_t st);
cudaError_t launch_prefix(const PrefixArgs& a, cudaStream_t st);
int decode_tile_tokens();
// Sets the message kv4_last_error_message() returns on this thread.
void set_error_message(const char* msg);
int decode_box_rows();

}  // namespace kv4
