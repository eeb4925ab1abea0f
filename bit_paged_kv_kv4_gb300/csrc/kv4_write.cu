// Quantise new K/V tokens into the paged 4-bit pool.
//
// NVFP4 ("SGLang's 4-bit KV cache", Figure 2 caption and "The 56% survives
// its own scale"): per 16-element block along the head dimension, an E4M3
// scale from the block maximum and the layer's FP32 global scale, and 16 E2M1
// codes.  INT4 per-token-head ("KV cache in 4 bits", "What we changed"): one
// FP32 scale per (token, head) row of K and of V, 4-bit two's-complement codes.
//
// The input is bf16 K/V, or FP8 E4M3 K/V with per-tensor scales (the form the
// engine hands to the cache in Figure 2): then each element is
// e4m3(code) * s_in, one FP32 product, and is encoded the same way.
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

// Quantise this thread's 8 elements x of row (token, head) and store them at
// (chunk, off).  NVFP4: the two threads of a 16-element block exchange their
// maxima; INT4: the D/8 threads of the row do.
template <int D, int FMT>
__device__ __forceinline__ void write_row_part(const WriteArgs& a, int kind, int part, const float (&x)[8],
                                               bool store, uint8_t* chunk, int off) {
  constexpr int TPR = D / 8;
  constexpr int RB = D / 2;
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(x[j]));
  if constexpr (FMT == KV4_NVFP4) {
    // block amax over the thread pair
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    const float g = __ldg(a.gscale + kind);
    const float sf = __fdiv_rn(amax, __fmul_rn(kE2M1Max, g));
    const uint32_t S = f32_to_e4m3(sf);
    const float denom = __fmul_rn(e4m3_to_f32(S), g);
    uint32_t word = 0;
    if (S != 0u && denom != 0.f) {
      const float rd = __frcp_rn(denom);
      float q[8];
      if (div_rn_in_range(rd, amax)) {
#pragma unroll
        for (int j = 0; j < 8; ++j) q[j] = div_rn_inrange(x[j], denom, rd);
      } else {                                  // operands near the FP32 range limits
#pragma unroll
        for (int j = 0; j < 8; ++j) q[j] = __fdiv_rn(x[j], denom);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) word |= f32x2_to_e2m1x2(q[2 * j], q[2 * j + 1]) << (8 * j);
    }
    constexpr int SB = D / 16;
    if (store && kind == 0) {
      *reinterpret_cast<uint32_t*>(chunk + static_cast<int64_t>(off) * RB + part * 4) = word;
      if ((part & 1) == 0)
        chunk[static_cast<int64_t>(a.P) * D + static_cast<int64_t>(off) * SB + (part >> 1)] =
            static_cast<uint8_t>(S);
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
      if ((part & 1) == 0)
        chunk[static_cast<int64_t>(a.P) * D + static_cast<int64_t>(a.P) * SB +
              static_cast<int64_t>(off >> 1) * 2 * SB + 2 * (part >> 1) + (off & 1)] = static_cast<uint8_t>(S);
    }
  } else if constexpr (FMT == KV4_FP8) {
    // FP8 per tensor: E4M3(x / s) for each element, s the layer's scale
    const float s = __ldg(a.gscale + kind);
    const float rs = __frcp_rn(s);
    float q[8];
    if (div_rn_in_range(rs, amax)) {
#pragma unroll
      for (int j = 0; j < 8; ++j) q[j] = div_rn_inrange(x[j], s, rs);
    } else {                                    // operands near the FP32 range limits
#pragma unroll
      for (int j = 0; j < 8; ++j) q[j] = __fdiv_rn(x[j], s);
    }
    if (store) {
      const uint32_t w0 = f32x2_to_e4m3x2(q[0], q[1]) | (f32x2_to_e4m3x2(q[2], q[3]) << 16);
      const uint32_t w1 = f32x2_to_e4m3x2(q[4], q[5]) | (f32x2_to_e4m3x2(q[6], q[7]) << 16);
      *reinterpret_cast<uint2*>(chunk + static_cast<int64_t>(kind) * a.P * D + static_cast<int64_t>(off) * D +
                                part * 8) = make_uint2(w0, w1);
    }
  } else {
    // row amax over the D/8 threads of the row (aligned groups of a warp)
#pragma unroll
    for (int o = 1; o < TPR; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = __fdiv_rn(amax, 7.0f);
    uint32_t word = 0;
    if (s != 0.f) {
      const float rs = __frcp_rn(s);
      float q[8];
      if (div_rn_in_range(rs, amax)) {
#pragma unroll
        for (int j = 0; j < 8; ++j) q[j] = div_rn_inrange(x[j], s, rs);
      } else {                                  // operands near the FP32 range limits
#pragma unroll
        for (int j = 0; j < 8; ++j) q[j] = __fdiv_rn(x[j], s);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        int c = __float2int_rn(q[j]);
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

// Thread (row (t, h), 8-element part, K|V = blockIdx.y).
template <int D, int FMT>
__global__ void __launch_bounds__(256)
write_kernel(const WriteArgs a) {
  grid_dep_launch();   // a following decode launch may be scheduled early
  constexpr int TPR = D / 8;                      // threads per row
  const uint32_t gtid = blockIdx.x * 256u + threadIdx.x;
  const int kind = blockIdx.y;                    // 0: K, 1: V
  const uint32_t row = gtid / TPR;
  const int part = static_cast<int>(gtid % TPR);
  const bool in_range = row < static_cast<uint32_t>(a.rows);
  const uint32_t t = in_range ? fdiv(row, a.hkv_div) : 0u;
  const int h = in_range ? static_cast<int>(row - t * static_cast<uint32_t>(a.Hkv)) : 0;

  // load 8 elements -> fp32 (rows past the end read row 0 and store nothing)
  const int64_t base = static_cast<int64_t>(in_range ? row : 0u) * D + part * 8;
  float x[8];
  if (a.k8 != nullptr) {
    // FP8 input: e4m3 (exact through f16) times the tensor's input scale
    const uint2 raw = __ldg(reinterpret_cast<const uint2*>((kind == 0 ? a.k8 : a.v8) + base));
    const float s_in = __ldg(a.in_scale + kind);
    uint32_t hh[4];
    e4m3x4_to_f16x2x2(raw.x, hh[0], hh[1]);
    e4m3x4_to_f16x2x2(raw.y, hh[2], hh[3]);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hh[j]));
      x[2 * j] = __fmul_rn(f.x, s_in);
      x[2 * j + 1] = __fmul_rn(f.y, s_in);
    }
  } else {
    const uint4 raw = __ldg(reinterpret_cast<const uint4*>((kind == 0 ? a.k : a.v) + base));
    const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float2 f = __bfloat1622float2(p2[j]);
      x[2 * j] = f.x;
      x[2 * j + 1] = f.y;
    }
  }
  // slots are below num_pages * P < 2^31 (the pool check), so 32-bit math
  const int64_t slot = in_range ? a.slot_mapping[t] : -1;
  const int64_t cap = static_cast<int64_t>(a.num_pages) * a.P;
  bool store = slot >= 0;
  if (slot >= cap) {
    if (part == 0) set_error(a.err, KV4_EBOUNDS);
    store = false;
  }
  const uint32_t su = store ? static_cast<uint32_t>(slot) : 0u;
  const uint32_t page = fdiv(su, a.p_div);
  const int off = static_cast<int>(su - page * static_cast<uint32_t>(a.P));
  uint8_t* chunk = a.pool + (static_cast<int64_t>(page) * a.Hkv + h) * a.chunk_bytes;
  write_row_part<D, FMT>(a, kind, part, x, store, chunk, off);
}

template <int D, int FMT>
static cudaError_t launch_write_t(const WriteArgs& a, cudaStream_t st) {
  const int64_t threads = static_cast<int64_t>(a.rows) * (D / 8);
  const int64_t blocks = (threads + 255) / 256;
  write_kernel<D, FMT><<<dim3(static_cast<unsigned>(blocks), 2), 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_write(const WriteArgs& a_in, cudaStream_t st) {
  if (a_in.T == 0) return cudaSuccess;
  WriteArgs a = a_in;
  a.rows = static_cast<int>(a.T * a.Hkv);
  a.hkv_div = make_fastdiv(static_cast<uint32_t>(a.Hkv));
  a.p_div = make_fastdiv(static_cast<uint32_t>(a.P));
  if (a.fmt == KV4_NVFP4) {
    switch (a.D) {
      case 64: return launch_write_t<64, KV4_NVFP4>(a, st);
      case 128: return launch_write_t<128, KV4_NVFP4>(a, st);
      default: return launch_write_t<256, KV4_NVFP4>(a, st);
    }
  }
  if (a.fmt == KV4_FP8) {
    switch (a.D) {
      case 64: return launch_write_t<64, KV4_FP8>(a, st);
      case 128: return launch_write_t<128, KV4_FP8>(a, st);
      default: return launch_write_t<256, KV4_FP8>(a, st);
    }
  }
  switch (a.D) {
    case 64: return launch_write_t<64, KV4_INT4_PTH>(a, st);
    case 128: return launch_write_t<128, KV4_INT4_PTH>(a, st);
    default: return launch_write_t<256, KV4_INT4_PTH>(a, st);
  }
}

}  // namespace kv4
