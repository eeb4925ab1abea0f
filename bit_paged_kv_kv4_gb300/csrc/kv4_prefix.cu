// Dequantise a cached 4-bit prefix into FP8 E4M3 workspaces: the first step
// of the chunked prefill / extend path of "SGLang's 4-bit KV cache", Figure 2,
// which turns the 4-bit prefix into FP8 in a buffer that is reused, then
// attends over prefix plus the current chunk.
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

__device__ __forceinline__ uint32_t pack_f16x2_same(__half h) {
  const uint32_t u = __half_as_ushort(h);
  return u | (u << 16);
}

// One E4M3 block of 16 elements of row (t, h): x_hat -> E4M3(x_hat / s8).
template <int D, int FMT>
__device__ __forceinline__ uint4 prefix_block(uint2 codes, float s, float g, float s8, float r8) {
  float xh[16];
  float bound;                                  // >= |x_hat| of every element
  if constexpr (FMT == KV4_NVFP4) {
    uint32_t h2[8];
    e2m1x8_to_f16x2x4(codes.x, *reinterpret_cast<uint32_t(*)[4]>(h2));
    e2m1x8_to_f16x2x4(codes.y, *reinterpret_cast<uint32_t(*)[4]>(h2 + 4));
    // e2m1 * e4m3 is exact in f16 (<= 6 significant bits, within [2^-10, 2688]),
    // so it equals the FP32 product; then one FP32 rounding for the * g
    const __half hs = __float2half_rn(s);     // s is an E4M3 value: exact
    const uint32_t s2 = pack_f16x2_same(hs);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t es = hmul2(h2[j], s2);
      const float2 e = __half22float2(*reinterpret_cast<const __half2*>(&es));
      xh[2 * j] = __fmul_rn(e.x, g);
      xh[2 * j + 1] = __fmul_rn(e.y, g);
    }
    bound = 6.f * s * g * 2.f;
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const uint32_t w = (j < 8) ? codes.x : codes.y;
      const int c = static_cast<int>((w >> (4 * (j & 7))) & 0xFu);
      xh[j] = __fmul_rn(static_cast<float>(c >= 8 ? c - 16 : c), s);
    }
    bound = 8.f * fabsf(s) * 2.f;
  }
  float q[16];
  if (r8 < 1.0e30f && bound * r8 < 1.0e30f) {
#pragma unroll
    for (int i = 0; i < 16; ++i) q[i] = div_rn_inrange(xh[i], s8, r8);
  } else {                                      // operands near the FP32 range limits
#pragma unroll
    for (int i = 0; i < 16; ++i) q[i] = __fdiv_rn(xh[i], s8);
  }
  uint32_t outw[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    outw[j] = f32x2_to_e4m3x2(q[4 * j], q[4 * j + 1]) | (f32x2_to_e4m3x2(q[4 * j + 2], q[4 * j + 3]) << 16);
  return make_uint4(outw[0], outw[1], outw[2], outw[3]);
}

// Thread (request b = blockIdx.z, K|V = blockIdx.y, row (t, h), blocks
// 2 part and 2 part + 1): 32 elements, so the per-thread set-up (indices,
// block-table lookup, reciprocal) is paid once per two blocks.
template <int D, int FMT>
__global__ void __launch_bounds__(256)
prefix_kernel(const PrefixArgs a) {
  constexpr int TPR = D / 32;                   // threads per row: 32 elements each
  constexpr int RB = D / 2, SB = D / 16;
  const int b = blockIdx.z;
  const int kind = blockIdx.y;
  const uint32_t gtid = blockIdx.x * 256u + threadIdx.x;
  const uint32_t row = gtid / TPR;              // (t, h), row < max_prefix_len * Hkv < 2^31
  const int part = static_cast<int>(gtid % TPR);
  const uint32_t t = fdiv(row, a.hkv_div);
  const int h = static_cast<int>(row - t * static_cast<uint32_t>(a.Hkv));
  int n = a.prefix_lens[b];
  const int cap = min(a.max_prefix_len, a.max_pages * a.P);
  if (n < 0 || n > cap) {
    if (gtid == 0) set_error(a.err, KV4_EBOUNDS);
    n = n < 0 ? 0 : cap;
  }
  if (t >= static_cast<uint32_t>(n)) return;

  const uint32_t pidx = fdiv(t, a.p_div);
  const int page = __ldg(a.block_table + static_cast<int64_t>(b) * a.max_pages + pidx);
  if (page < 0 || page >= a.num_pages) {
    if (part == 0) set_error(a.err, KV4_EBOUNDS);
    return;
  }
  const int off = static_cast<int>(t - pidx * static_cast<uint32_t>(a.P));
  const uint8_t* chunk = a.pool + (static_cast<int64_t>(page) * a.Hkv + h) * a.chunk_bytes;
  uint2 codes[2];
  float sc[2];
  if (FMT == KV4_NVFP4 && kind == 1) {
    // V is stored in token pairs: byte d of pair row off/2 holds element d of
    // this token in nibble off%2.  Gather the blocks' 32 nibbles back into
    // the packed order (element 2j in the low nibble of byte j).
    const uint4* src = reinterpret_cast<const uint4*>(
        chunk + static_cast<int64_t>(a.P) * RB + static_cast<int64_t>(off >> 1) * D + part * 32);
    const int sh = 4 * (off & 1);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const uint4 w = src[k];
      const uint32_t x0 = (w.x >> sh) & 0x0F0F0F0Fu, x1 = (w.y >> sh) & 0x0F0F0F0Fu;
      const uint32_t x2 = (w.z >> sh) & 0x0F0F0F0Fu, x3 = (w.w >> sh) & 0x0F0F0F0Fu;
      // byte pairs (n_2j, n_2j+1) -> one byte each, then keep bytes 0 and 2
      codes[k].x = prmt(x0 | (x0 >> 4), x1 | (x1 >> 4), 0x6420u);
      codes[k].y = prmt(x2 | (x2 >> 4), x3 | (x3 >> 4), 0x6420u);
    }
  } else {
    const uint4 w = *reinterpret_cast<const uint4*>(
        chunk + static_cast<int64_t>(kind) * a.P * RB + static_cast<int64_t>(off) * RB + part * 16);
    codes[0] = make_uint2(w.x, w.y);
    codes[1] = make_uint2(w.z, w.w);
  }
  if constexpr (FMT == KV4_NVFP4) {
    // K: one scale row per token; V: pair rows, byte 2*blk + off%2
    if (kind == 0) {
      const uint8_t* sp = chunk + static_cast<int64_t>(a.P) * D + static_cast<int64_t>(off) * SB + 2 * part;
      sc[0] = e4m3_to_f32(sp[0]);
      sc[1] = e4m3_to_f32(sp[1]);
    } else {
      const uint8_t* sp = chunk + static_cast<int64_t>(a.P) * D + static_cast<int64_t>(a.P) * SB +
                          static_cast<int64_t>(off >> 1) * 2 * SB + 4 * part + (off & 1);
      sc[0] = e4m3_to_f32(sp[0]);
      sc[1] = e4m3_to_f32(sp[2]);
    }
  } else {
    sc[0] = sc[1] = *reinterpret_cast<const float*>(chunk + static_cast<int64_t>(a.P) * D +
                                                    (static_cast<int64_t>(kind) * a.P + off) * 4);
  }
  const float s8 = __ldg(a.fp8_scale + kind);
  const float r8 = __frcp_rn(s8);
  const float g = (FMT == KV4_NVFP4) ? __ldg(a.gscale + kind) : 1.f;
  const int64_t orow = a.cu_prefix[b] + t;
  uint4* dst = reinterpret_cast<uint4*>((kind == 0 ? a.out_k : a.out_v) + (orow * a.Hkv + h) * D + part * 32);
  dst[0] = prefix_block<D, FMT>(codes[0], sc[0], g, s8, r8);
  dst[1] = prefix_block<D, FMT>(codes[1], sc[1], g, s8, r8);
}

template <int D, int FMT>
static cudaError_t launch_prefix_t(const PrefixArgs& a, cudaStream_t st) {
  const int64_t threads = static_cast<int64_t>(a.max_prefix_len) * a.Hkv * (D / 32);
  const int64_t blocks = (threads + 255) / 256;
  prefix_kernel<D, FMT><<<dim3(static_cast<unsigned>(blocks), 2, a.B), 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_prefix(const PrefixArgs& a_in, cudaStream_t st) {
  const int64_t threads = static_cast<int64_t>(a_in.max_prefix_len) * a_in.Hkv * (a_in.D / 16);
  if (threads == 0 || a_in.B == 0) return cudaSuccess;
  PrefixArgs a = a_in;
  a.hkv_div = make_fastdiv(static_cast<uint32_t>(a.Hkv));
  a.p_div = make_fastdiv(static_cast<uint32_t>(a.P));
  if (a.fmt == KV4_NVFP4) {
    switch (a.D) {
      case 64: return launch_prefix_t<64, KV4_NVFP4>(a, st);
      case 128: return launch_prefix_t<128, KV4_NVFP4>(a, st);
      default: return launch_prefix_t<256, KV4_NVFP4>(a, st);
    }
  }
  switch (a.D) {
    case 64: return launch_prefix_t<64, KV4_INT4_PTH>(a, st);
    case 128: return launch_prefix_t<128, KV4_INT4_PTH>(a, st);
    default: return launch_prefix_t<256, KV4_INT4_PTH>(a, st);
  }
}

}  // namespace kv4
