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
// A unit is one 16-element block (one NVFP4 scale block) of the same
// head-dim range of two consecutive tokens 2p and 2p+1 of the call; D/16
// neighbouring units form a row (INT4 reduces its row maximum over their
// threads).  The grid is sized to the resident CTAs and each warp walks its
// 32 units a grid apart, staging their input bytes and slots in the warp's
// part of a shared-memory ring with asynchronous copies (cp.async) issued
// kWriteStages - 1 steps ahead, so the loads of later units are in flight
// while the current ones are encoded; the lanes copy 512 contiguous input
// bytes an instruction for one another.
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
#include "kv4_encode.cuh"
#include "kv4_internal.h"

namespace kv4 {

// E2M1 codes of 16 quotients, element 2j in the low nibble of byte j.
__device__ __forceinline__ uint2 e2m1x16(const float (&q)[16]) {
  return make_uint2(f32x8_to_e2m1x8(q), f32x8_to_e2m1x8(q + 8));
}

// Eight codes of token 2p (nibble i of a) and of token 2p+1 (nibble i of b)
// -> the pair row's eight bytes a_i | b_i << 4 (element i in byte i).
__device__ __forceinline__ uint2 zip_nibbles(uint32_t a, uint32_t b) {
  const uint32_t ev = (a & 0x0F0F0F0Fu) | ((b << 4) & 0xF0F0F0F0u);     // elements 0, 2, 4, 6
  const uint32_t od = ((a >> 4) & 0x0F0F0F0Fu) | (b & 0xF0F0F0F0u);     // elements 1, 3, 5, 7
  return make_uint2(prmt(ev, od, 0x5140u), prmt(ev, od, 0x7362u));
}
__device__ __forceinline__ uint4 zip16(uint2 a, uint2 b) {
  const uint2 lo = zip_nibbles(a.x, b.x), hi = zip_nibbles(a.y, b.y);
  return make_uint4(lo.x, lo.y, hi.x, hi.y);
}

// q_j = RN(x_j / b) for 16 values given their negations nx_j = -x_j, b > 0
// with yb = RN(1/b): Markstein's correction step on FP32 pairs where
// div_rn_in_range(yb, amax) holds (amax >= every |x_j|), else the IEEE
// division.  With ny = -yb the step reads q0 = RN(nx ny) = RN(x yb),
// e = b q0 + nx = -(x - b q0) (exact under fma), q = RN(e ny + q0)
// = RN(q0 + (x - b q0) yb): the same bits as the usual order, and for x = -0
// (nx = +0) it gives q = -0, the IEEE sign of a zero quotient, with no
// fix-up.
__device__ __forceinline__ void div16(const float (&nx)[16], float b, float yb, float amax, float (&q)[16]) {
  if (div_rn_in_range(yb, amax)) {
    const uint64_t b2 = f2(b, b), ny2 = f2(-yb, -yb);
#pragma unroll
    for (int j = 0; j < 16; j += 2) {
      const uint64_t x = f2(nx[j], nx[j + 1]);
      const uint64_t q0 = mul_f2(x, ny2);
      const uint64_t e = fma_f2(b2, q0, x);
      f2_split(fma_f2(e, ny2, q0), q[j], q[j + 1]);
    }
  } else {                                      // operands near the FP32 range limits
#pragma unroll
    for (int j = 0; j < 16; ++j) q[j] = -__fdiv_rn(nx[j], b);
  }
}

// Eight packed nibbles (element i in nibble i) -> eight bytes, nibble i in
// the low half of byte i.
__device__ __forceinline__ uint2 spread_nibbles(uint32_t w) {
  const uint32_t lo4 = w & 0x0F0F0F0Fu, hi4 = (w >> 4) & 0x0F0F0F0Fu;
  return make_uint2(prmt(lo4, hi4, 0x5140u), prmt(lo4, hi4, 0x7362u));
}

constexpr int kWriteThreads = 256;
constexpr int kWriteWarps = kWriteThreads / 32;
constexpr int kWriteStages = 2;          // steps staged per warp (one in flight while one is encoded)
constexpr int kWriteCtasPerSm = 3;       // 3 x 41 KB of staging per SM
// A warp's stage: 128 16-byte data slots (its 32 units x 2 tokens x 32 bf16
// bytes; FP8 input uses the first 64), then 32 slot pairs (16 bytes a unit).
constexpr uint32_t kWarpData = 128 * 16;
constexpr uint32_t kWarpStage = kWarpData + 32 * 16;
constexpr int kWriteSmem = kWriteStages * kWriteWarps * kWarpStage;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// bf16 data slot m = 64 j + 2 l + c (token j, unit lane l, 16-byte half c)
// sits at slot m ^ bit 3 of m: the copies (32 consecutive m an instruction)
// and the reads (m = 2l + c over the lanes) are both free of bank conflicts.
__device__ __forceinline__ uint32_t slot_pos(uint32_t m) { return m ^ ((m >> 3) & 1u); }

// Unit u -> (first token t0 = 2p, head h, block b).
struct Unit {
  int64_t t0;
  int h, b;
};
template <int D>
__device__ __forceinline__ Unit unit_of(const WriteArgs& a, uint32_t u) {
  constexpr int NB = D / 16;
  const uint32_t ph = u / NB;                     // (pair, head)
  const uint32_t pair = fdiv(ph, a.hkv_div);
  return Unit{2 * static_cast<int64_t>(pair), static_cast<int>(ph - pair * static_cast<uint32_t>(a.Hkv)),
              static_cast<int>(u % NB)};
}

// Stage the input and slots of the warp's units ub + 0..31 at `wst` (the
// warp's stage).  bf16: copy instruction k moves data slots m = 32 k + lane,
// i.e. half (lane & 1) of unit 16 (k & 1) + lane / 2's block of token k / 2,
// so each instruction reads 512 contiguous bytes of a row run; FP8: slot
// 32 j + lane is token j of the lane's own unit.  Slots: the even lane of a
// pair copies token t0's slot, the odd lane t0 + 1's.  Nothing is copied for
// a unit past the end or a token past T (those bytes are never stored).
template <int D>
__device__ __forceinline__ void stage_warp(const WriteArgs& a, int kind, uint32_t ub, uint32_t lane,
                                           uint32_t wst) {
  if (a.k8 != nullptr) {
    const uint32_t u = ub + lane;
    if (u >= a.units) return;
    const Unit n = unit_of<D>(a, u);
    const uint8_t* src = (kind == 0 ? a.k8 : a.v8) + 16 * n.b;
    const int64_t row0 = n.t0 * a.Hkv + n.h;
    cp_async16(wst + 16 * lane, src + row0 * D);
    if (n.t0 + 1 < a.T) cp_async16(wst + 16 * (32 + lane), src + (row0 + a.Hkv) * D);
    cp_async8(wst + kWarpData + 16 * lane, a.slot_mapping + n.t0);
    if (n.t0 + 1 < a.T) cp_async8(wst + kWarpData + 16 * lane + 8, a.slot_mapping + n.t0 + 1);
    return;
  }
  const __nv_bfloat16* src = kind == 0 ? a.k : a.v;
  const uint32_t c = lane & 1u;
#pragma unroll
  for (int q = 0; q < 2; ++q) {                   // unit lane l = 16 q + lane / 2
    const uint32_t l = 16 * q + (lane >> 1), u = ub + l;
    if (u >= a.units) continue;
    const Unit n = unit_of<D>(a, u);
    const __nv_bfloat16* p = src + (n.t0 * a.Hkv + n.h) * D + 16 * n.b + 8 * c;
    const bool live1 = n.t0 + 1 < a.T;
    cp_async16(wst + 16 * slot_pos(2 * l + c), p);
    if (live1) cp_async16(wst + 16 * slot_pos(64 + 2 * l + c), p + static_cast<int64_t>(a.Hkv) * D);
    if (c == 0 || live1) cp_async8(wst + kWarpData + 16 * l + 8 * c, a.slot_mapping + n.t0 + c);
  }
}

// -x as FP32 for the two bf16 values x of w (exact): (w << 16) + 2^31 and
// (w & 0xFFFF0000) ^ 2^31, one integer instruction each (written as PTX so
// that they are not turned into float negations, which the packed FP32
// operations that consume them cannot fold).
__device__ __forceinline__ void neg_bf16x2(uint32_t w, float& lo, float& hi) {
  uint32_t l, h;
  asm("mad.lo.u32 %0, %1, 65536, 0x80000000;" : "=r"(l) : "r"(w));
  asm("lop3.b32 %0, %1, 0xFFFF0000, 0x80000000, 0x6a;" : "=r"(h) : "r"(w));
  lo = __uint_as_float(l);
  hi = __uint_as_float(h);
}

// The negated 16 elements of token j (0: t0, 1: t0 + 1) of unit lane `lane`
// staged at `wst` -> FP32: -bf16 (exact), or E4M3 times -s_in as one FP32
// product (the negation of RN(e4m3 * s_in)).
__device__ __forceinline__ void staged16_neg(const WriteArgs& a, int kind, uint32_t wst, uint32_t lane, int j,
                                             float (&nx)[16]) {
  if (a.k8 != nullptr) {
    const uint4 raw = lds128(wst + 16 * (32 * j + lane));
    const float ns_in = -__ldg(a.in_scale + kind);
    const uint64_t ns2 = f2(ns_in, ns_in);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t hh[2];
      e4m3x4_to_f16x2x2(w[i], hh[0], hh[1]);
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hh[k]));   // exact
        f2_split(mul_f2(f2(f.x, f.y), ns2), nx[4 * i + 2 * k], nx[4 * i + 2 * k + 1]);
      }
    }
  } else {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const uint4 raw = lds128(wst + 16 * slot_pos(64 * j + 2 * lane + u));
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) neg_bf16x2(w[k], nx[8 * u + 2 * k], nx[8 * u + 2 * k + 1]);
    }
  }
}

// The 16 elements of one token already loaded (bf16: raw[0..1]; FP8: raw[0])
// -> their negations in FP32, as staged16_neg computes them.
__device__ __forceinline__ void raw16_neg(const WriteArgs& a, int kind, const uint4 (&raw)[2], float (&nx)[16]) {
  if (a.k8 != nullptr) {
    const float ns_in = -__ldg(a.in_scale + kind);
    const uint64_t ns2 = f2(ns_in, ns_in);
    const uint32_t w[4] = {raw[0].x, raw[0].y, raw[0].z, raw[0].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t hh[2];
      e4m3x4_to_f16x2x2(w[i], hh[0], hh[1]);
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hh[k]));   // exact
        f2_split(mul_f2(f2(f.x, f.y), ns2), nx[4 * i + 2 * k], nx[4 * i + 2 * k + 1]);
      }
    }
  } else {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const uint32_t w[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) neg_bf16x2(w[k], nx[8 * u + 2 * k], nx[8 * u + 2 * k + 1]);
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
__device__ __forceinline__ Dest dest_of(const WriteArgs& a, int64_t t, int64_t slot, int h, bool flag) {
  Dest d{nullptr, 0, -1, false};
  if (t >= a.T || slot < 0) return d;
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

// Encode unit u (K|V = kind) from the warp's stage `wst`; `live` false for a
// thread past the last unit (it computes on whatever the stage holds and
// stores nothing, so that whole rows of threads share the INT4 shuffles).
template <int D, int FMT, int kind, bool direct = false>
__device__ __forceinline__ void write_unit(const WriteArgs& a, uint32_t u, bool live, uint32_t wst, uint32_t lane,
                                           const float2* s_den, float g6, float r6) {
  constexpr int NB = D / 16;                      // threads per row
  constexpr int RB = D / 2, SB = D / 16;
  const Unit n = unit_of<D>(a, u);
  const int b = n.b, h = n.h;
  const int64_t t0 = live ? n.t0 : a.T;           // past the end: no destination
  // token k's destination (taken after the arithmetic where that keeps
  // fewer registers live across it)
  // direct: both tokens' input words and slots are loaded here, before any
  // arithmetic, so that a small call pays one memory round trip
  uint4 raw[2][2];
  int64_t dslot[2] = {-1, -1};
  if constexpr (direct) {
    const int64_t row0 = n.t0 * a.Hkv + h;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int64_t e = ((n.t0 + k < a.T) ? row0 + k * a.Hkv : row0) * D + 16 * b;
      if (a.k8 != nullptr) {
        raw[k][0] = __ldg(reinterpret_cast<const uint4*>((kind == 0 ? a.k8 : a.v8) + e));
      } else {
        const uint4* src = reinterpret_cast<const uint4*>((kind == 0 ? a.k : a.v) + e);
        raw[k][0] = __ldg(src);
        raw[k][1] = __ldg(src + 1);
      }
      if (t0 + k < a.T) dslot[k] = __ldg(a.slot_mapping + t0 + k);
    }
  }
  auto dest = [&](int k) {
    int64_t slot = -1;
    if constexpr (direct) {
      slot = dslot[k];
    } else {
      const uint2 sl = lds64(wst + kWarpData + 16 * lane + 8 * k);
      slot = static_cast<int64_t>((static_cast<uint64_t>(sl.y) << 32) | sl.x);
    }
    return dest_of(a, t0 + k, slot, h, b == 0);
  };
  // token k's 16 elements, negated, from the stage or (direct) from global memory
  auto elems = [&](int k, float (&x)[16]) {
    if constexpr (direct) {
      raw16_neg(a, kind, raw[k], x);
    } else {
      staged16_neg(a, kind, wst, lane, k, x);
    }
  };

  // each token's elements are read from the stage as their negations
  if constexpr (FMT == KV4_NVFP4) {
    uint32_t S[2];
    uint2 kw[2];                      // token k's codes, element i in nibble i
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      float x[16];
      elems(k, x);
      float amax = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(x[j]));
      const float sf = div_rn(amax, g6, r6);
      S[k] = f32_to_e4m3(sf);
      const float2 dr = s_den[S[k]];
      kw[k] = make_uint2(0u, 0u);
      if (S[k] != 0u && dr.x != 0.f) {
        float q[16];
        div16(x, dr.x, dr.y, amax, q);
        kw[k] = e2m1x16(q);
      }
    }
    const Dest d0 = dest(0), d1 = dest(1);
    if constexpr (kind == 0) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const Dest& d = k == 0 ? d0 : d1;
        if (!d.ok) continue;
        *reinterpret_cast<uint2*>(d.chunk + static_cast<int64_t>(d.off) * RB + 8 * b) = kw[k];
        d.chunk[static_cast<int64_t>(a.P) * D + static_cast<int64_t>(d.off) * SB + b] = static_cast<uint8_t>(S[k]);
      }
    } else if (d0.ok && d1.ok && (d0.slot & 1) == 0 && d1.slot == d0.slot + 1) {
      // both halves of one pair row: byte d = element d of token 2p (low
      // nibble) and of token 2p+1 (high nibble); scale bytes (s_even, s_odd)
      *reinterpret_cast<uint4*>(d0.chunk + static_cast<int64_t>(a.P) * RB + static_cast<int64_t>(d0.off >> 1) * D +
                                16 * b) = zip16(kw[0], kw[1]);
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
          const uint2 sp = spread_nibbles(u == 0 ? kw[k].x : kw[k].y);
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
      float x[16];
      elems(k, x);
      const Dest d = dest(k);
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
  } else if constexpr (kind == 0) {
    // K: token rows, each token stored as soon as it is encoded
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      float x[16];
      elems(k, x);
      const Dest d = dest(k);
      // row amax over the D/16 threads of the row (aligned groups of a warp)
      float amax = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(x[j]));
#pragma unroll
      for (int o = 1; o < NB; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      const float s = div7(amax);
      uint2 word = make_uint2(0u, 0u);
      if (s != 0.f) {
        const float rs = __frcp_rn(s);
        float q[16];
        div16(x, s, rs, amax, q);
        word = make_uint2(int4x8(q), int4x8(q + 8));
      }
      if (d.ok) {
        *reinterpret_cast<uint2*>(d.chunk + static_cast<int64_t>(d.off) * RB + 8 * b) = word;
        if (b == 0) reinterpret_cast<float*>(d.chunk + static_cast<int64_t>(a.P) * D)[d.off] = s;
      }
    }
  } else {
    // V: both tokens encoded, then stored into their pair rows
    uint2 word[2];                    // token k's codes, element i in nibble i
    float sc[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      float x[16];
      elems(k, x);
      // row amax over the D/16 threads of the row (aligned groups of a warp)
      float amax = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(x[j]));
#pragma unroll
      for (int o = 1; o < NB; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      const float s = div7(amax);
      word[k] = make_uint2(0u, 0u);
      if (s != 0.f) {
        const float rs = __frcp_rn(s);
        float q[16];
        div16(x, s, rs, amax, q);
        word[k] = make_uint2(int4x8(q), int4x8(q + 8));
      }
      sc[k] = s;
    }
    const Dest d0 = dest(0), d1 = dest(1);
    auto put_scale = [&](const Dest& d, float s) {
      if (b == 0) reinterpret_cast<float*>(d.chunk + static_cast<int64_t>(a.P) * D)[a.P + d.off] = s;
    };
    if (d0.ok && d1.ok && (d0.slot & 1) == 0 && d1.slot == d0.slot + 1) {
      // both tokens of one pair row: word 4b + c holds 16-bit chunk c
      // (elements 4c .. 4c+3 of this block) of token 2p low, of 2p+1 high
      *reinterpret_cast<uint4*>(d0.chunk + static_cast<int64_t>(a.P) * RB + static_cast<int64_t>(d0.off >> 1) * D +
                                16 * b) =
          make_uint4(prmt(word[0].x, word[1].x, 0x5410u), prmt(word[0].x, word[1].x, 0x7632u),
                     prmt(word[0].y, word[1].y, 0x5410u), prmt(word[0].y, word[1].y, 0x7632u));
      put_scale(d0, sc[0]);
      put_scale(d1, sc[1]);
    } else {
      // a token alone in its pair row (in this thread): its own 16-bit
      // halves, bytes no other token writes, one 2-byte store each
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const Dest& d = k == 0 ? d0 : d1;
        if (!d.ok) continue;
        uint16_t* dst = reinterpret_cast<uint16_t*>(d.chunk + static_cast<int64_t>(a.P) * RB +
                                                    static_cast<int64_t>(d.off >> 1) * D + 16 * b + 2 * (d.off & 1));
        dst[0] = static_cast<uint16_t>(word[k].x);
        dst[2] = static_cast<uint16_t>(word[k].x >> 16);
        dst[4] = static_cast<uint16_t>(word[k].y);
        dst[6] = static_cast<uint16_t>(word[k].y >> 16);
        put_scale(d, sc[k]);
      }
    }
  }
}

// Each warp walks units a grid apart (K|V = kind), staging kWriteStages - 1
// steps ahead of the one it encodes; a lane may copy bytes another lane
// reads, so the warp syncs after its copies land and before a stage is
// refilled.
template <int D, int FMT, int kind>
__device__ __forceinline__ void write_walk(const WriteArgs& a, uint8_t* s_stage, const float2* s_den, float g6,
                                           float r6) {
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  const uint32_t total = a.units, stride = gridDim.x * kWriteThreads;
  const uint32_t w0 = smem_u32(s_stage) + warp * kWarpStage;
  constexpr uint32_t kStageBytes = kWriteWarps * kWarpStage;
  uint32_t ub = blockIdx.x * kWriteThreads + warp * 32;      // the warp's units are ub + lane
#pragma unroll
  for (int s = 0; s < kWriteStages - 1; ++s) {
    if (ub + s * stride < total) stage_warp<D>(a, kind, ub + s * stride, lane, w0 + s * kStageBytes);
    cp_async_commit();
  }
  int cur = 0;
  for (; ub < total; ub += stride) {
    const uint32_t ahead = ub + (kWriteStages - 1) * stride;
    const int nxt = cur == 0 ? kWriteStages - 1 : cur - 1;     // the stage encoded last
    __syncwarp();                                 // every lane is done reading it
    if (ahead < total) stage_warp<D>(a, kind, ahead, lane, w0 + nxt * kStageBytes);
    cp_async_commit();
    cp_async_wait<kWriteStages - 1>();            // this lane's copies for step ub
    __syncwarp();                                 // and every other lane's
    const uint32_t u = ub + lane;
    write_unit<D, FMT, kind>(a, u < total ? u : 0u, u < total, w0 + cur * kStageBytes, lane, s_den, g6, r6);
    cur = cur + 1 == kWriteStages ? 0 : cur + 1;
  }
  cp_async_wait<0>();                             // no copy outlives the CTA
}

// Persistent CTAs of kWriteThreads threads, kWriteCtasPerSm per SM, half on
// K (blockIdx.y = 0) and half on V; each warp walks units a grid apart.  A
// call whose units fit one thread each (a decode step's new tokens) takes
// the direct form instead: one unit a thread, loaded straight from global
// memory, no staging (and no dynamic shared memory).
template <int D, int FMT, bool direct>
__global__ void __launch_bounds__(kWriteThreads, kWriteCtasPerSm)
write_kernel(const WriteArgs a) {
  grid_dep_launch();   // a following decode launch may be scheduled early
  grid_dep_wait();     // launched early itself: inputs of the previous kernel are visible from here
  const int kind = blockIdx.y;                    // 0: K, 1: V
  extern __shared__ __align__(16) uint8_t s_stage[];
  // NVFP4: (denominator, its reciprocal) of every E4M3 block-scale byte S:
  // denom = RN(e4m3(S) * g), 1/denom correctly rounded
  __shared__ float2 s_den[FMT == KV4_NVFP4 ? 256 : 1];
  float g6 = 1.f, r6 = 1.f;
  if constexpr (FMT == KV4_NVFP4) {
    const float g = __ldg(a.gscale + kind);
    g6 = __fmul_rn(kE2M1Max, g);
    r6 = __frcp_rn(g6);
    const float den = __fmul_rn(e4m3_to_f32(threadIdx.x), g);
    s_den[threadIdx.x] = make_float2(den, __frcp_rn(den));
    __syncthreads();
  }
  if constexpr (direct) {
    const uint32_t u = blockIdx.x * kWriteThreads + threadIdx.x;
    const bool live = u < a.units;
    if (kind == 0) write_unit<D, FMT, 0, true>(a, live ? u : 0u, live, 0u, 0u, s_den, g6, r6);
    else write_unit<D, FMT, 1, true>(a, live ? u : 0u, live, 0u, 0u, s_den, g6, r6);
  } else {
    if (kind == 0) write_walk<D, FMT, 0>(a, s_stage, s_den, g6, r6);
    else write_walk<D, FMT, 1>(a, s_stage, s_den, g6, r6);
  }
}

// Launched with programmatic stream serialisation: the kernel may be
// scheduled while the previous kernel on the stream drains, and reads
// nothing before its grid_dep_wait().
template <typename K>
static cudaError_t launch_pdl_write(K* k, dim3 grid, size_t smem, cudaStream_t st, const WriteArgs& a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kWriteThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, a);
}

template <int D, int FMT>
static cudaError_t launch_write_t(const WriteArgs& a, cudaStream_t st) {
  const int64_t need = (static_cast<int64_t>(a.units) + kWriteThreads - 1) / kWriteThreads;
  const int64_t resident = static_cast<int64_t>(a.sms) * kWriteCtasPerSm / 2;   // per K|V
  if (need <= resident)                         // one unit a thread
    return launch_pdl_write(write_kernel<D, FMT, true>, dim3(static_cast<unsigned>(need), 2), 0, st, a);
  auto* k = write_kernel<D, FMT, false>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kWriteSmem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  return launch_pdl_write(k, dim3(static_cast<unsigned>(resident > 0 ? resident : 1), 2), kWriteSmem, st, a);
}

cudaError_t launch_write(const WriteArgs& a_in, cudaStream_t st) {
  if (a_in.T == 0) return cudaSuccess;
  WriteArgs a = a_in;
  a.rows = static_cast<int>(a.T * a.Hkv);
  a.units = static_cast<uint32_t>((a.T + 1) / 2 * a.Hkv * (a.D / 16));
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
