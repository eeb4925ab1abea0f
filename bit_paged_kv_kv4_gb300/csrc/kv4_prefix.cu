// Dequantise a cached 4-bit prefix into FP8 E4M3 workspaces: the chunked
// prefill / extend path of "SGLang's 4-bit KV cache", Figure 2, which "reads
// NVFP4 and dequantizes the cached prefix into a reused FP8 workspace" before
// attending over prefix plus the current chunk.
//
// One thread turns 16 consecutive head-dim elements (one NVFP4 block) of one
// (token, head, K|V) row into 16 E4M3 bytes: x_hat = (e2m1 * e4m3) * g in
// FP32 (NVFP4) or code * s (INT4), then E4M3(x_hat / s_fp8) with RNE and
// saturation; the division is the correctly rounded div_rn.  Pure streaming:
// one code load (8 bytes; 16 for the token-pair rows of NVFP4 V, of which
// this token's nibbles are kept), one scale, one 16-byte store.
#include <cstdint>

#include "kv4_device.cuh"
#include "kv4_internal.h"

namespace kv4 {

__global__ void __launch_bounds__(256)
prefix_kernel(const PrefixArgs a) {
  const int D = a.D;
  const int tpr = D / 16;                      // threads per row: 16 elements each
  const int b = blockIdx.z;
  const int kind = blockIdx.y;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t row = tid / tpr;               // (t, h)
  const int part = static_cast<int>(tid % tpr);
  const int t = static_cast<int>(row / a.Hkv);
  const int h = static_cast<int>(row % a.Hkv);
  int n = a.prefix_lens[b];
  const int cap = min(a.max_prefix_len, a.max_pages * a.P);
  if (n < 0 || n > cap) {
    if (tid == 0) set_error(a.err, KV4_EBOUNDS);
    n = n < 0 ? 0 : cap;
  }
  if (t >= n) return;

  int page = __ldg(a.block_table + static_cast<int64_t>(b) * a.max_pages + t / a.P);
  if (page < 0 || page >= a.num_pages) {
    if (part == 0) set_error(a.err, KV4_EBOUNDS);
    return;
  }
  const int off = t % a.P;
  const uint8_t* chunk = a.pool + (static_cast<int64_t>(page) * a.Hkv + h) * a.chunk_bytes;
  const int RB = D / 2;
  uint2 codes;
  if (a.fmt == KV4_NVFP4 && kind == 1) {
    // V is stored in token pairs: byte d of pair row off/2 holds element d of
    // this token in nibble off%2.  Gather the block's 16 nibbles back into
    // the packed order (element 2j in the low nibble of byte j).
    const uint4 w = *reinterpret_cast<const uint4*>(
        chunk + static_cast<int64_t>(a.P) * RB + static_cast<int64_t>(off >> 1) * D + part * 16);
    const int sh = 4 * (off & 1);
    const uint32_t x0 = (w.x >> sh) & 0x0F0F0F0Fu, x1 = (w.y >> sh) & 0x0F0F0F0Fu;
    const uint32_t x2 = (w.z >> sh) & 0x0F0F0F0Fu, x3 = (w.w >> sh) & 0x0F0F0F0Fu;
    // byte pairs (n_2j, n_2j+1) -> one byte each, then keep bytes 0 and 2
    codes.x = prmt(x0 | (x0 >> 4), x1 | (x1 >> 4), 0x6420u);
    codes.y = prmt(x2 | (x2 >> 4), x3 | (x3 >> 4), 0x6420u);
  } else {
    codes = *reinterpret_cast<const uint2*>(
        chunk + static_cast<int64_t>(kind) * a.P * RB + static_cast<int64_t>(off) * RB + part * 8);
  }
  const float s8 = __ldg(a.fp8_scale + kind);
  const float r8 = __frcp_rn(s8);

  float xh[16];
  if (a.fmt == KV4_NVFP4) {
    const int SB = D / 16;
    // K: one scale row per token; V: pair rows, byte 2*blk + off%2
    const uint8_t* sc = (kind == 0)
        ? chunk + static_cast<int64_t>(a.P) * D + static_cast<int64_t>(off) * SB + part
        : chunk + static_cast<int64_t>(a.P) * D + static_cast<int64_t>(a.P) * SB +
              static_cast<int64_t>(off >> 1) * 2 * SB + 2 * part + (off & 1);
    const float s = e4m3_to_f32(*sc);          // one block of 16 per thread
    const float g = __ldg(a.gscale + kind);
    uint32_t h2[8];
    e2m1x8_to_f16x2x4(codes.x, *reinterpret_cast<uint32_t(*)[4]>(h2));
    e2m1x8_to_f16x2x4(codes.y, *reinterpret_cast<uint32_t(*)[4]>(h2 + 4));
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float2 e = __half22float2(*reinterpret_cast<const __half2*>(&h2[j]));
      xh[2 * j] = __fmul_rn(__fmul_rn(e.x, s), g);
      xh[2 * j + 1] = __fmul_rn(__fmul_rn(e.y, s), g);
    }
  } else {
    const float s = *reinterpret_cast<const float*>(chunk + static_cast<int64_t>(a.P) * D +
                                                     (static_cast<int64_t>(kind) * a.P + off) * 4);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const uint32_t w = (j < 8) ? codes.x : codes.y;
      const int c = static_cast<int>((w >> (4 * (j & 7))) & 0xFu);
      xh[j] = __fmul_rn(static_cast<float>(c >= 8 ? c - 16 : c), s);
    }
  }
  uint32_t outw[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    outw[j] = f32x2_to_e4m3x2(div_rn(xh[4 * j], s8, r8), div_rn(xh[4 * j + 1], s8, r8)) |
              (f32x2_to_e4m3x2(div_rn(xh[4 * j + 2], s8, r8), div_rn(xh[4 * j + 3], s8, r8)) << 16);
  const int64_t orow = a.cu_prefix[b] + t;
  uint8_t* dst = (kind == 0 ? a.out_k : a.out_v) + (orow * a.Hkv + h) * D + part * 16;
  *reinterpret_cast<uint4*>(dst) = make_uint4(outw[0], outw[1], outw[2], outw[3]);
}

cudaError_t launch_prefix(const PrefixArgs& a, cudaStream_t st) {
  const int64_t threads = static_cast<int64_t>(a.max_prefix_len) * a.Hkv * (a.D / 16);
  if (threads == 0 || a.B == 0) return cudaSuccess;
  const int bs = 256;
  const int64_t blocks = (threads + bs - 1) / bs;
  prefix_kernel<<<dim3(static_cast<unsigned>(blocks), 2, a.B), bs, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace kv4
