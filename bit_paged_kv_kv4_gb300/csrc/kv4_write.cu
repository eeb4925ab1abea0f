// Quantise new K/V tokens into the paged 4-bit pool.
//
// NVFP4 ("SGLang's 4-bit KV cache", Figure 2 caption and "The 56% survives
// its own scale"): per 16-element block along the head dimension, an E4M3
// scale from the block maximum and the layer's FP32 global scale, and 16 E2M1
// codes.  INT4 per-token-head ("KV cache in 4 bits", "What we changed"): one
// FP32 scale per (token, head) row of K and of V, 4-bit two's-complement codes.
//
// One thread owns 8 consecutive elements (one 16-byte load of bf16); two
// neighbouring threads form an NVFP4 block, D/8 neighbouring threads a row.
// NVFP4 V goes to the token-pair rows the decode kernel reads (element d of
// tokens 2p and 2p+1 share a byte); K and INT4 rows are one per token.
// All encoder arithmetic is IEEE FP32 with round-to-nearest (no fast-math),
// in the order the header states, so the bytes match the oracle exactly; the
// per-element divisions by the block's (or row's) scale use a correctly
// rounded reciprocal-and-correction division (div_rn), which returns the same
// value as the IEEE quotient.
#include <cstdint>

#include "kv4_device.cuh"
#include "kv4_internal.h"

namespace kv4 {

__global__ void __launch_bounds__(256)
write_kernel(const WriteArgs a) {
  grid_dep_launch();   // a following decode launch may be scheduled early
  const int D = a.D;
  const int tpr = D / 8;                          // threads per row
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int kind = blockIdx.y;                    // 0: K, 1: V
  const int64_t rows = a.T * a.Hkv;
  const int64_t row = tid / tpr;
  const int part = static_cast<int>(tid % tpr);
  const bool in_range = row < rows;
  const int64_t t = in_range ? row / a.Hkv : 0;
  const int h = in_range ? static_cast<int>(row % a.Hkv) : 0;

  // load 8 bf16 -> fp32 (rows past the end read row 0 and store nothing)
  const __nv_bfloat16* src = (kind == 0 ? a.k : a.v) + (in_range ? row : 0) * D + part * 8;
  uint4 raw = __ldg(reinterpret_cast<const uint4*>(src));
  float x[8];
  {
    const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float2 f = __bfloat1622float2(p2[j]);
      x[2 * j] = f.x;
      x[2 * j + 1] = f.y;
    }
  }
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(x[j]));

  const int64_t slot = in_range ? a.slot_mapping[t] : -1;
  const int64_t cap = static_cast<int64_t>(a.num_pages) * a.P;
  bool store = slot >= 0;
  if (slot >= cap) {
    if (part == 0) set_error(a.err, KV4_EBOUNDS);
    store = false;
  }
  const int64_t page = store ? slot / a.P : 0;
  const int off = store ? static_cast<int>(slot % a.P) : 0;
  uint8_t* chunk = a.pool + (page * a.Hkv + h) * a.chunk_bytes;
  const int RB = D / 2;

  if (a.fmt == KV4_NVFP4) {
    // block amax over the thread pair
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    const float g = __ldg(a.gscale + kind);
    const float sf = __fdiv_rn(amax, __fmul_rn(kE2M1Max, g));
    const uint32_t S = f32_to_e4m3(sf);
    const float denom = __fmul_rn(e4m3_to_f32(S), g);
    uint32_t word = 0;
    if (S != 0u && denom != 0.f) {
      const float rd = __frcp_rn(denom);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t byte = f32x2_to_e2m1x2(div_rn(x[2 * j], denom, rd),
                                              div_rn(x[2 * j + 1], denom, rd));
        word |= byte << (8 * j);
      }
    }
    if (store && kind == 0) {
      uint8_t* codes = chunk + static_cast<int64_t>(off) * RB;
      *reinterpret_cast<uint32_t*>(codes + part * 4) = word;
      if ((part & 1) == 0) {
        const int SB = D / 16;
        uint8_t* sc = chunk + static_cast<int64_t>(a.P) * D + static_cast<int64_t>(off) * SB;
        sc[part >> 1] = static_cast<uint8_t>(S);
      }
    } else if (store) {
      // V rows are stored in token pairs: byte d of pair row off/2 holds element
      // d of the even token (low nibble) and of the odd token (high nibble).
      // This token's 8 elements go to 8 consecutive bytes, in its own nibbles;
      // the partner token may be written concurrently, so the update is an
      // atomic clear and set of those nibbles only.
      const uint32_t lo4 = word & 0x0F0F0F0Fu, hi4 = (word >> 4) & 0x0F0F0F0Fu;
      const uint64_t spread = (static_cast<uint64_t>(prmt(lo4, hi4, 0x7362u)) << 32) | prmt(lo4, hi4, 0x5140u);
      const int sh = 4 * (off & 1);
      unsigned long long* dst = reinterpret_cast<unsigned long long*>(
          chunk + static_cast<int64_t>(a.P) * RB + static_cast<int64_t>(off >> 1) * D + part * 8);
      atomicAnd(dst, ~(0x0F0F0F0F0F0F0F0Full << sh));
      atomicOr(dst, static_cast<unsigned long long>(spread << sh));
      if ((part & 1) == 0) {
        const int SB = D / 16;
        uint8_t* sc = chunk + static_cast<int64_t>(a.P) * D + static_cast<int64_t>(a.P) * SB +
                      static_cast<int64_t>(off >> 1) * 2 * SB;
        sc[2 * (part >> 1) + (off & 1)] = static_cast<uint8_t>(S);
      }
    }
  } else {
    // row amax over the D/8 threads of the row (aligned groups of a warp)
    for (int o = 1; o < tpr; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = __fdiv_rn(amax, 7.0f);
    uint32_t word = 0;
    if (s != 0.f) {
      const float rs = __frcp_rn(s);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        int c = __float2int_rn(div_rn(x[j], s, rs));
        c = c < -8 ? -8 : (c > 7 ? 7 : c);
        word |= (static_cast<uint32_t>(c) & 0xFu) << (4 * j);
      }
    }
    if (store) {
      uint8_t* codes = chunk + static_cast<int64_t>(kind) * a.P * RB + static_cast<int64_t>(off) * RB;
      *reinterpret_cast<uint32_t*>(codes + part * 4) = word;
      if (part == 0) {
        float* sc = reinterpret_cast<float*>(chunk + static_cast<int64_t>(a.P) * D) +
                    static_cast<int64_t>(kind) * a.P + off;
        *sc = s;
      }
    }
  }
}

cudaError_t launch_write(const WriteArgs& a, cudaStream_t st) {
  const int64_t threads = a.T * a.Hkv * (a.D / 8);
  if (threads == 0) return cudaSuccess;
  const int bs = 256;
  const int64_t blocks = (threads + bs - 1) / bs;
  write_kernel<<<dim3(static_cast<unsigned>(blocks), 2), bs, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace kv4
