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
// One thread owns one 16-element block (one NVFP4 scale block) of the same
// head-dim range of two consecutive tokens 2p and 2p+1 of the call; D/16
// neighbouring threads form a row (INT4 reduces its row maximum over them).
// NVFP4 V goes to the token-pair rows the decode kernel reads (element d of
// tokens 2p and 2p+1 share a byte): when the two tokens land in the two
// halves of one pair row (the usual prefill), the thread writes the pair's
// bytes with plain stores; otherwise each token's nibbles are set with an
// atomic clear and set (its partner may be written by another thread).  K,
// INT4 and FP8 rows are one per token.  All encoder arithmetic is IEEE FP32
// with round-to-nearest (no fast-math), in the order the header states, so
// the bytes match the oracle exactly; the per-element divisions use a
// correctly rounded reciprocal-and-correction division (div_rn), which
// returns the same value as the IEEE quotient, with the reciprocals of the
// 256 possible block-scale denominators taken once per CTA.
#include <cstdint>

#include "kv4_device.cuh"
#include "kv4_internal.h"

namespace kv4 {

// E2M1 codes of 16 quotients, element 2j in the low nibble of byte j.
__device__ __forceinline__ uint2 e2m1x16(const float (&q)[16]) {
  return make_uint2(f32x8_to_e2m1x8(q), f32x8_to_e2m1x8(q + 8));
}

// q_j = RN(x_j / b) for 16 values, b > 0 with yb = RN(1/b): div_rn on FP32
// pairs where div_rn_in_range(yb, amax) holds (amax >= every |x_j|), else
// the IEEE division.
__device__ __forceinline__ void div16(const float (&x)[16], float b, float yb, float amax, float (&q)[16]) {
  if (div_rn_in_range(yb, amax)) {
    const uint64_t nb = f2(-b, -b), yb2 = f2(yb, yb);
#pragma unroll
    for (int j = 0; j < 16; j += 2) div_rn_pair(x[j], x[j + 1], nb, yb2, q[j], q[j + 1]);
  } else {                                      // operands near the FP32 range limits
#pragma unroll
    for (int j = 0; j < 16; ++j) q[j] = __fdiv_rn(x[j], b);
  }
}

// Eight packed nibbles (element i in nibble i) -> eight bytes, nibble i in
// the low half of byte i.
__device__ __forceinline__ uint2 spread_nibbles(uint32_t w) {
  const uint32_t lo4 = w & 0x0F0F0F0Fu, hi4 = (w >> 4) & 0x0F0F0F0Fu;
  return make_uint2(prmt(lo4, hi4, 0x5140u), prmt(lo4, hi4, 0x7362u));
}

// 16 consecutive elements of row `row` of K or V -> FP32 (bf16, or E4M3
// times the input scale as one FP32 product).
__device__ __forceinline__ void load16(const WriteArgs& a, int kind, int64_t row, int D, int b, float (&x)[16]) {
  const int64_t base = row * D + 16 * b;
  if (a.k8 != nullptr) {
    const uint4 raw = __ldg(reinterpret_cast<const uint4*>((kind == 0 ? a.k8 : a.v8) + base));
    const float s_in = __ldg(a.in_scale + kind);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t hh[2];
      e4m3x4_to_f16x2x2(w[i], hh[0], hh[1]);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hh[j]));
        x[4 * i + 2 * j] = __fmul_rn(f.x, s_in);
        x[4 * i + 2 * j + 1] = __fmul_rn(f.y, s_in);
      }
    }
  } else {
    const uint4* src = reinterpret_cast<const uint4*>((kind == 0 ? a.k : a.v) + base);
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const uint4 raw = __ldg(src + u);
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        x[8 * u + 2 * j] = __uint_as_float(w[j] << 16);           // bf16 -> FP32 is exact
        x[8 * u + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
      }
    }
  }
}

// Where token t goes: its chunk and offset, or nothing (slot < 0, or past
// the pool, which is recorded).
struct Dest {
  uint8_t* chunk;
  int off;
  int64_t slot;
  bool ok;
};
__device__ __forceinline__ Dest dest_of(const WriteArgs& a, int64_t t, int h, bool flag) {
  Dest d{nullptr, 0, -1, false};
  if (t >= a.T) return d;
  const int64_t slot = a.slot_mapping[t];
  if (slot < 0) return d;
  if (slot >= static_cast<int64_t>(a.num_pages) * a.P) {
    if (flag) set_error(a.err, KV4_EBOUNDS);
    return d;
  }
  // slots are below num_pages * P < 2^31 (the pool check), so 32-bit math
  const uint32_t su = static_cast<uint32_t>(slot);
  const uint32_t page = fdiv(su, a.p_div);
  d.off = static_cast<int>(su - page * static_cast<uint32_t>(a.P));
  d.chunk = a.pool + (static_cast<int64_t>(page) * a.Hkv + h) * a.chunk_bytes;
  d.slot = slot;
  d.ok = true;
  return d;
}

// Thread (token pair p, head h, 16-element block b; K|V = blockIdx.y).
template <int D, int FMT>
__global__ void __launch_bounds__(256, 4)
write_kernel(const WriteArgs a) {
  grid_dep_launch();   // a following decode launch may be scheduled early
  constexpr int NB = D / 16;                      // threads per row
  constexpr int RB = D / 2, SB = D / 16;
  const int kind = blockIdx.y;                    // 0: K, 1: V
  // NVFP4: (denominator, its reciprocal) of every E4M3 block-scale byte S:
  // denom = RN(e4m3(S) * g), 1/denom correctly rounded
  __shared__ float2 s_den[FMT == KV4_NVFP4 ? 256 : 1];
  float g = 1.f, g6 = 1.f, r6 = 1.f;
  if constexpr (FMT == KV4_NVFP4) {
    g = __ldg(a.gscale + kind);
    g6 = __fmul_rn(kE2M1Max, g);
    r6 = __frcp_rn(g6);
    const float den = __fmul_rn(e4m3_to_f32(threadIdx.x), g);
    s_den[threadIdx.x] = make_float2(den, __frcp_rn(den));
    __syncthreads();
  }
  const uint32_t gtid = blockIdx.x * 256u + threadIdx.x;
  const uint32_t ph = gtid / NB;                  // (pair, head)
  const int b = static_cast<int>(gtid % NB);
  const uint32_t pair = fdiv(ph, a.hkv_div);
  const int h = static_cast<int>(ph - pair * static_cast<uint32_t>(a.Hkv));
  const int64_t t0 = 2 * static_cast<int64_t>(pair);
  // rows past the end compute on row 0 and store nothing (whole rows of
  // threads share the shuffles below)
  const bool live0 = t0 < a.T, live1 = t0 + 1 < a.T;
  const Dest d0 = dest_of(a, t0, h, b == 0), d1 = dest_of(a, t0 + 1, h, b == 0);

  float x0[16], x1[16];
  load16(a, kind, live0 ? t0 * a.Hkv + h : 0, D, b, x0);
  load16(a, kind, live1 ? (t0 + 1) * a.Hkv + h : 0, D, b, x1);

  if constexpr (FMT == KV4_NVFP4) {
    uint2 word[2];
    uint32_t S[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float(&x)[16] = k == 0 ? x0 : x1;
      float amax = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(x[j]));
      const float sf = div_rn(amax, g6, r6);
      S[k] = f32_to_e4m3(sf);
      const float2 dr = s_den[S[k]];
      word[k] = make_uint2(0u, 0u);
      if (S[k] != 0u && dr.x != 0.f) {
        float q[16];
        div16(x, dr.x, dr.y, amax, q);
        word[k] = e2m1x16(q);
      }
    }
    if (kind == 0) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const Dest& d = k == 0 ? d0 : d1;
        if (!d.ok) continue;
        *reinterpret_cast<uint2*>(d.chunk + static_cast<int64_t>(d.off) * RB + 8 * b) = word[k];
        d.chunk[static_cast<int64_t>(a.P) * D + static_cast<int64_t>(d.off) * SB + b] = static_cast<uint8_t>(S[k]);
      }
    } else if (d0.ok && d1.ok && (d0.slot & 1) == 0 && d1.slot == d0.slot + 1) {
      // both halves of one pair row: byte d = element d of token 2p (low
      // nibble) and of token 2p+1 (high nibble); scale bytes (s_even, s_odd)
      const uint2 a0 = spread_nibbles(word[0].x), a1 = spread_nibbles(word[0].y);
      const uint2 b0 = spread_nibbles(word[1].x), b1 = spread_nibbles(word[1].y);
      *reinterpret_cast<uint4*>(d0.chunk + static_cast<int64_t>(a.P) * RB + static_cast<int64_t>(d0.off >> 1) * D +
                                16 * b) =
          make_uint4(a0.x | (b0.x << 4), a0.y | (b0.y << 4), a1.x | (b1.x << 4), a1.y | (b1.y << 4));
      *reinterpret_cast<uint16_t*>(d0.chunk + static_cast<int64_t>(a.P) * D + static_cast<int64_t>(a.P) * SB +
                                   static_cast<int64_t>(d0.off >> 1) * 2 * SB + 2 * b) =
          static_cast<uint16_t>(S[0] | (S[1] << 8));
    } else {
      // a token alone in its pair row (in this thread): an atomic clear and
      // set of its own nibbles, since the partner may be written concurrently
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const Dest& d = k == 0 ? d0 : d1;
        if (!d.ok) continue;
        const int sh = 4 * (d.off & 1);
        unsigned long long* dst = reinterpret_cast<unsigned long long*>(
            d.chunk + static_cast<int64_t>(a.P) * RB + static_cast<int64_t>(d.off >> 1) * D + 16 * b);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const uint2 sp = spread_nibbles(u == 0 ? word[k].x : word[k].y);
          const uint64_t v = (static_cast<uint64_t>(sp.y) << 32) | sp.x;
          atomicAnd(dst + u, ~(0x0F0F0F0F0F0F0F0Full << sh));
          atomicOr(dst + u, static_cast<unsigned long long>(v << sh));
        }
        d.chunk[static_cast<int64_t>(a.P) * D + static_cast<int64_t>(a.P) * SB +
                static_cast<int64_t>(d.off >> 1) * 2 * SB + 2 * b + (d.off & 1)] = static_cast<uint8_t>(S[k]);
      }
    }
  } else if constexpr (FMT == KV4_FP8) {
    // FP8 per tensor: E4M3(x / s) for each element, s the layer's scale
    const float s = __ldg(a.gscale + kind);
    const float rs = __frcp_rn(s);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float(&x)[16] = k == 0 ? x0 : x1;
      const Dest& d = k == 0 ? d0 : d1;
      float amax = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(x[j]));
      float q[16];
      div16(x, s, rs, amax, q);
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        w[i] = f32x2_to_e4m3x2(q[4 * i], q[4 * i + 1]) | (f32x2_to_e4m3x2(q[4 * i + 2], q[4 * i + 3]) << 16);
      if (d.ok)
        *reinterpret_cast<uint4*>(d.chunk + static_cast<int64_t>(kind) * a.P * D + static_cast<int64_t>(d.off) * D +
                                  16 * b) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float(&x)[16] = k == 0 ? x0 : x1;
      const Dest& d = k == 0 ? d0 : d1;
      // row amax over the D/16 threads of the row (aligned groups of a warp)
      float amax = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(x[j]));
#pragma unroll
      for (int o = 1; o < NB; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      const float s = __fdiv_rn(amax, 7.0f);
      uint2 word = make_uint2(0u, 0u);
      if (s != 0.f) {
        const float rs = __frcp_rn(s);
        float q[16];
        div16(x, s, rs, amax, q);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          int c = __float2int_rn(q[j]);
          c = c < -8 ? -8 : (c > 7 ? 7 : c);
          (j < 8 ? word.x : word.y) |= (static_cast<uint32_t>(c) & 0xFu) << (4 * (j & 7));
        }
      }
      if (d.ok) {
        uint8_t* codes = d.chunk + static_cast<int64_t>(kind) * a.P * RB + static_cast<int64_t>(d.off) * RB;
        *reinterpret_cast<uint2*>(codes + 8 * b) = word;
        if (b == 0)
          reinterpret_cast<float*>(d.chunk + static_cast<int64_t>(a.P) * D)[static_cast<int64_t>(kind) * a.P + d.off] = s;
      }
    }
  }
}

template <int D, int FMT>
static cudaError_t launch_write_t(const WriteArgs& a, cudaStream_t st) {
  const int64_t threads = (a.T + 1) / 2 * a.Hkv * (D / 16);
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
