// Device-side building blocks for libkv4 (sm_103a): FP4/FP8 conversions,
// the f16 tensor-core MMA, mbarriers, TMA / bulk copies and the shared
// memory swizzle the TMA writes.  Inline PTX only; no library kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include "../../include/kv4.h"
#include "kv4_internal.h"

namespace kv4 {

// ---------------------------------------------------------------- constants
constexpr int kBlock = 16;            // NVFP4 elements per E4M3 block scale
constexpr float kE2M1Max = 6.0f;

// A bounded wait gives up after this many SM clock cycles (about one second
// at GB300 clocks) and records KV4_ETIMEOUT instead of spinning forever.
constexpr long long kWaitCycles = 2000000000LL;

// Records the first failure in the per-device error word; never traps.
__device__ __forceinline__ void set_error(int* err, int code) {
  if (err != nullptr) atomicCAS(err, 0, code);
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialisation may start before the previous kernel on the stream has
// finished; grid_dep_wait() blocks until that kernel has completed and its
// memory is visible (a no-op for a normally launched kernel).
// grid_dep_launch() lets the next such kernel be scheduled early; it still
// waits in its own grid_dep_wait() for this grid to complete.
__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------ conversions
// Two FP32 values -> one byte of two E2M1 codes, round to nearest even,
// saturating at 6, sign kept: `lo` goes to the low nibble.
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
      "cvt.u16.u8 %0, t;\n\t}"
      : "=h"(r) : "f"(hi), "f"(lo));
  return r & 0xFFu;
}

// FP32 -> E4M3 code, round to nearest even, saturating at 448.
__device__ __forceinline__ uint32_t f32_to_e4m3(float x) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(x));
  return r & 0xFFu;
}

// Two FP32 -> two E4M3 codes in one 16-bit value (`lo` in the low byte).
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two E4M3 codes (16 bits, low byte first) -> f16x2, exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t r;
  uint16_t t = static_cast<uint16_t>(two);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(t));
  return r;
}

// E4M3 code -> FP32, exact.
__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
  uint32_t h2 = e4m3x2_to_f16x2(code & 0xFFu);
  return __half2float(__ushort_as_half(static_cast<uint16_t>(h2 & 0xFFFFu)));
}

// One byte of two E2M1 codes -> f16x2 (low nibble -> low half), exact.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t r;
  uint16_t t = static_cast<uint16_t>(byte & 0xFFu);
  asm("{\n\t.reg .b8 b;\n\t"
      "cvt.u8.u16 b, %1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b;\n\t}"
      : "=r"(r) : "h"(t));
  return r;
}

// Four bytes of E2M1 code pairs -> four f16x2 (byte i -> r[i], low nibble ->
// low half), exact.  Unpacking the word into byte registers in one PTX block
// lets each conversion read its byte directly (no separate extraction).
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t (&r)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(w));
}

// Two pairs of E4M3 codes (16-bit halves of `w`) -> two f16x2, exact:
// r0 = (w.byte0, w.byte1), r1 = (w.byte2, w.byte3).
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& r0, uint32_t& r1) {
  asm("{\n\t.reg .b16 h0, h1;\n\t"
      "mov.b32 {h0, h1}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, h0;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, h1;\n\t}"
      : "=r"(r0), "=r"(r1) : "r"(w));
}

// E2M1 code (low nibble) -> FP32, exact.
__device__ __forceinline__ float e2m1_to_f32(uint32_t code) {
  uint32_t h2 = e2m1x2_to_f16x2(code & 0xFu);
  return __half2float(__ushort_as_half(static_cast<uint16_t>(h2 & 0xFFFFu)));
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

__device__ __forceinline__ uint32_t lop3_and_xor(uint32_t a, uint32_t mask, uint32_t x) {
  // (a & mask) ^ x
  return (a & mask) ^ x;
}

// ------------------------------------------------------------ tensor core
// D = A(16x16, f16, row) * B(16x8, f16, col) + C, FP32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 matrix of 16-bit elements held one row pair per thread
// (thread t: row t/4, columns 2(t%4), 2(t%4)+1) -> the same layout of the
// transposed matrix.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t r;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

// ------------------------------------------------------------ shared memory
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds8(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

// Byte offset inside a tile of rows of RB bytes written by a TMA load with
// the matching swizzle (RB = 128: 128B, 64: 64B, 32: 32B swizzle): the 16-byte
// unit index is XORed with address bits 7.. of the row start.  The tile must
// start at a multiple of the swizzle span (1024/512/256 bytes).
template <int RB>
__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t col) {
  constexpr uint32_t M = (RB == 128) ? 7u : (RB == 64) ? 3u : 1u;
  const uint32_t o = row * RB;
  return o + (col ^ (((o >> 7) & M) << 4));
}

// ------------------------------------------------------------ mbarriers
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
               :: "r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}
// Bounded wait for phase `parity` of a barrier: false if it ran out of time.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitCycles) return false;
  }
  return true;
}

// ------------------------------------------------------------ TMA / bulk
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 2-D tiled TMA load of box {x extent, y extent} at (x, y) into shared
// memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x,
                                            int y, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar),
         "l"(policy)
      : "memory");
}

// 3-D tiled TMA load of box {x, y, z extents} at (x, y, z) into shared memory
// (box laid out z-major, then y, then x), completing on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar),
         "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                            int w, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar),
         "l"(policy)
      : "memory");
}

// Contiguous bulk copy global -> shared (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;"
      :: "r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// n / f.d for n < 2^31 (see FastDiv).
__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv& f) {
  return (__umulhi(n, f.m) + n) >> f.s;
}

// ------------------------------------------------------------ division
// a / b rounded to nearest even, given yb = __frcp_rn(b) (1/b correctly
// rounded).  Markstein's theorem (P. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1),
// 1990): q0 = RN(a * yb) is within one ulp of a/b, the residual a - b*q0 is
// exact under a fused multiply-add, and RN(q0 + residual * yb) equals
// RN(a/b) whenever no intermediate overflows or underflows.  Outside that
// range (a reciprocal that is subnormal or not finite, a first quotient that
// is not finite) it falls back to the IEEE division; a quotient that falls
// below FP32's normal range may be off in its last subnormal bit, which no
// caller sees (it converts to a zero of E4M3 or E2M1).  The sign of a zero quotient follows a (as a/b with
// b > 0 does).  Callers only pass b > 0.
__device__ __forceinline__ float div_rn(float a, float b, float yb) {
  const float q0 = __fmul_rn(a, yb);
  if (!(fabsf(q0) < 1.0e30f) || !(yb < 1.0e30f) || !(yb >= 1.17549435e-38f)) return __fdiv_rn(a, b);
  const float r = __fmaf_rn(-b, q0, a);
  return copysignf(__fmaf_rn(r, yb, q0), a);
}

// div_rn without the range check, for callers that have checked once, with
// div_rn_in_range(yb, bound), that yb is a normal number below 1e30 and that
// |a * yb| < 1e30 for every a they pass (|a| <= bound).
__device__ __forceinline__ bool div_rn_in_range(float yb, float bound) {
  return yb < 1.0e30f && yb >= 1.17549435e-38f && bound * yb < 1.0e30f;
}
__device__ __forceinline__ float div_rn_inrange(float a, float b, float yb) {
  const float q0 = __fmul_rn(a, yb);
  const float r = __fmaf_rn(-b, q0, a);
  return copysignf(__fmaf_rn(r, yb, q0), a);
}

// Packed FP32 pairs: each lane of mul.rn / fma.rn .f32x2 is the IEEE
// round-to-nearest result of the scalar operation, so pairs give the same
// bits as two scalar instructions at half the issue cost.
__device__ __forceinline__ uint64_t f2(float x, float y) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
  return r;
}
__device__ __forceinline__ void f2_split(uint64_t v, float& x, float& y) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(v));
}
__device__ __forceinline__ uint64_t mul_f2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t fma_f2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// RN(a / b) for a pair (div_rn_inrange on each lane, Markstein's correction
// step): q0 = a yb, r = a - b q0 (exact under fma), q = q0 + r yb; the sign of
// a zero quotient follows a.  nb = (-b, -b), yb2 = (yb, yb) with yb = RN(1/b).
__device__ __forceinline__ void div_rn_pair(float a0, float a1, uint64_t nb, uint64_t yb2, float& q0o,
                                            float& q1o) {
  const uint64_t a = f2(a0, a1);
  const uint64_t q0 = mul_f2(a, yb2);
  const uint64_t r = fma_f2(nb, q0, a);
  f2_split(fma_f2(r, yb2, q0), q0o, q1o);
  q0o = __uint_as_float((__float_as_uint(q0o) & 0x7FFFFFFFu) | (__float_as_uint(a0) & 0x80000000u));
  q1o = __uint_as_float((__float_as_uint(q1o) & 0x7FFFFFFFu) | (__float_as_uint(a1) & 0x80000000u));
}

// Eight FP32 values -> eight E2M1 codes, element i in nibble i.
__device__ __forceinline__ uint32_t f32x8_to_e2m1x8(const float* q) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(q[0]), "f"(q[1]), "f"(q[2]), "f"(q[3]), "f"(q[4]), "f"(q[5]), "f"(q[6]), "f"(q[7]));
  return r;
}

// ------------------------------------------------------------ misc
__device__ __forceinline__ float fast_log2(float x) {
  float r;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float fast_exp2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

}  // namespace kv4
