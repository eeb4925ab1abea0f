// Encoder pieces shared by the pool writes (kv4_write.cu, kv4_k8v4.cu): the
// INT4 row scale and codes, bit-exact with the IEEE FP32 definitions.
#pragma once
#include <cstdint>

#include "kv4_device.cuh"

namespace kv4 {

// RN(a / 7) for a >= 0 as the IEEE division gives it: Markstein's correction
// step with RN(1/7) where a lies in [1e-30, 1e30) (quotient and residual
// normal, no overflow), else the IEEE division (0, tiny, huge, non-finite).
__device__ __forceinline__ float div7(float a) {
  if (a >= 1.0e-30f && a < 1.0e30f) {
    const float y = 0.142857149f;                 // RN(1/7)
    const float q0 = __fmul_rn(a, y);
    return __fmaf_rn(__fmaf_rn(-7.0f, q0, a), y, q0);
  }
  return __fdiv_rn(a, 7.0f);
}

// INT4 codes of eight quotients q (|q| < 7.5 here: q = x / RN(amax / 7) with
// |x| <= amax, so no code leaves [-7, 7] and no clamp is needed), element i
// in nibble i: q + 1.5 * 2^23, rounded to nearest even, holds rint(q) in its
// low mantissa bits (two's complement modulo 16), as __float2int_rn would
// round it.  The additions run on FP32 pairs.
__device__ __forceinline__ uint32_t int4x8(const float* q) {
  const uint64_t m2 = f2(12582912.0f, 12582912.0f);
  uint32_t by[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint64_t t;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(t) : "l"(f2(q[2 * k], q[2 * k + 1])), "l"(m2));
    float t0, t1;
    f2_split(t, t0, t1);
    // byte k = nibble(t0) | nibble(t1) << 4 (higher bits are not used)
    by[k] = (__float_as_uint(t0) & 0xFu) + __float_as_uint(t1) * 16u;
  }
  return prmt(prmt(by[0], by[1], 0x0040u), prmt(by[2], by[3], 0x0040u), 0x5410u);
}

}  // namespace kv4
