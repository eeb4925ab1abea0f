// The k8v4 variant ("SGLang's 4-bit KV cache", section "Against what this
// site already established": the other 4-bit KV cache of the month keeps
// keys in FP8 and values in 4 bits and gives both one fixed FP32 Hadamard
// rotation of size D).  H = S_D / sqrt(D) (Sylvester), symmetric and
// orthogonal.
//
// Write (k8v4_write_kernel): D/32 lanes per (token, head) row of K or V.
// The row is rotated in FP32 by the fast Walsh-Hadamard transform, stages
// len = 1, 2, ..., D/2 replacing (x_i, x_{i+len}) by (x_i + x_{i+len},
// x_i - x_{i+len}) (i with bit len clear), then scaled by float32(1/sqrt D);
// a lane holds 32 consecutive elements for stages below 32, then (after a
// transpose through shared memory) one position of each 32-element block
// for the others.  Keys: E4M3(k_rot / s_K) (one
// per-tensor FP32 scale); values: INT4 per row, s = amax / 7,
// code = clamp(rne(v_rot / s), -8, 7).  IEEE FP32 throughout, so the bytes
// match the test oracle's; the divisions take Markstein's correction step
// (the IEEE quotient) and the INT4 codes the round-to-nearest-even magic
// addition, as in kv4_write.cu.
// Chunk of P tokens: [K codes P*D][V codes P*D/2][V scales FP32 * P], the V
// codes in token-pair rows by 16-bit halves as in the INT4 pool.
//
// Decode runs the NVFP4 / INT4 decode kernel (kv4_decode4.cu) with FP8 keys:
// q is rotated the same way (q_rot . k_rot = q . k), the softmax runs over
// the dequantised rotated keys, and the combine rotates the merged output
// back (H H = I).
#include <cstdint>

#include "kv4_device.cuh"
#include "kv4_encode.cuh"
#include "kv4_internal.h"

namespace kv4 {
namespace {


template <int D>
__device__ __forceinline__ float inv_sqrt_d() {
  return D == 64 ? 0.125f : (D == 128 ? 0.08838834764831845f : 0.0625f);
}

// ---------------------------------------------------------------- write
// A row of D elements is held by LPR = D / 32 consecutive lanes, 32
// consecutive elements a lane (a warp holds RPW = 32 / LPR rows), so stages
// len = 1 .. 16 of the transform stay in the lane.  The row then goes
// through shared memory once, transposed: afterwards a lane holds, for every
// one of the row's LPR blocks of 32 elements, the same NL = 32 / LPR
// positions inside the block, so stages len = 32 .. D/2 (which pair equal
// positions of different blocks) stay in the lane too.  The butterflies run
// on FP32 pairs (add / sub .f32x2: each lane the IEEE RN result), so the
// bits are those of scalar stages in the same order.
//
// Transpose layout: per row D floats, block b (the elements lane b of the
// row held) at 128 b bytes, its 16-byte chunk c at chunk c ^ (writer lane &
// 7).  A lane reads chunks [NC rl, NC rl + NC) of every block, NC = 8 / LPR,
// in an order rotated by its row's place in the warp; together the two
// make every store and load phase of eight lanes hit eight distinct bank
// groups at D = 64, 128 and 256.
__device__ __forceinline__ uint64_t add_f2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t sub_f2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// (x[i], x[i+1]), (x[j], x[j+1]) -> their sums and differences, in place
__device__ __forceinline__ void butterfly2(float* x, int i, int j) {
  const uint64_t p = f2(x[i], x[i + 1]), q = f2(x[j], x[j + 1]);
  f2_split(add_f2(p, q), x[i], x[i + 1]);
  f2_split(sub_f2(p, q), x[j], x[j + 1]);
}

// INT4 codes of four quotients (|q| < 7.5), element i in nibble i: the
// magic addition of int4x8, for half as many.
__device__ __forceinline__ uint32_t int4x4(const float* q) {
  const uint64_t m2 = f2(12582912.0f, 12582912.0f);
  uint32_t by[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    float t0, t1;
    f2_split(add_f2(f2(q[2 * k], q[2 * k + 1]), m2), t0, t1);
    by[k] = (__float_as_uint(t0) & 0xFu) + __float_as_uint(t1) * 16u;
  }
  return prmt(by[0], by[1], 0x0040u) & 0xFFFFu;
}

// RN(x / b) for a pair from the negated dividends nx = -x (Markstein's
// correction step with both signs flipped): q0 = RN(nx ny), e = fma(b, q0,
// nx) = -(x - b q0) (exact), q = RN(e ny + q0), with ny = -RN(1/b).  The
// result is the IEEE quotient x / b, the sign of a zero quotient included,
// with no fix-up.  bb = (b, b), ny2 = (ny, ny).
__device__ __forceinline__ void div_rn_pair_neg(float nx0, float nx1, uint64_t bb, uint64_t ny2, float& q0o,
                                                float& q1o) {
  const uint64_t nx = f2(nx0, nx1);
  const uint64_t q0 = mul_f2(nx, ny2);
  const uint64_t e = fma_f2(bb, q0, nx);
  f2_split(fma_f2(e, ny2, q0), q0o, q1o);
}

template <int D>
__global__ void __launch_bounds__(256) k8v4_write_kernel(const K8V4WriteArgs a) {
  constexpr int E = 32;                                   // elements per lane
  constexpr int LPR = D / E;                              // lanes per row
  constexpr int RPW = 32 / LPR;                           // rows per warp
  constexpr int NC = 8 / LPR;                             // chunks of a block a lane reads back
  constexpr int NL = 4 * NC;                              // elements of a block a lane holds
  static_assert(LPR >= 2 && LPR <= 8, "head dim 64, 128 or 256");
  __shared__ __align__(16) float s_rows[8][RPW * D];      // a warp's rows (4 KB)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rl = lane % LPR, rw = lane / LPR;             // place in the row, row in the warp
  const int64_t row = (static_cast<int64_t>(blockIdx.x) * 8 + warp) * RPW + rw;
  const int kind = blockIdx.y;                            // 0: K, 1: V
  // rows past the end compute on row 0 and store nothing (lanes of a row
  // share the transpose and the shuffles below, and rows of a warp share the
  // warp)
  const bool live = row < a.rows;
  const int64_t r0 = live ? row : 0;
  // rows < 2^31 (host check): 32-bit multiply-high division by Hkv
  const uint32_t t32 = fdiv(static_cast<uint32_t>(r0), a.hkv_div);
  const int64_t t = t32;
  const int h = static_cast<int>(static_cast<uint32_t>(r0) - t32 * static_cast<uint32_t>(a.Hkv));
  const int64_t slot = live ? a.slot_mapping[t] : -1;     // issued early; used at the store

  // E consecutive bf16 -> FP32
  const uint4* src = reinterpret_cast<const uint4*>((kind == 0 ? a.k : a.v) + r0 * D + rl * E);
  float x[E];
#pragma unroll
  for (int u = 0; u < E / 8; ++u) {
    const uint4 w = __ldg(src + u);
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[8 * u + 2 * j] = __uint_as_float(ww[j] << 16);        // bf16 -> FP32 is exact
      x[8 * u + 2 * j + 1] = __uint_as_float(ww[j] & 0xFFFF0000u);
    }
  }
  // FWHT stages len = 1 .. 16 in the lane: len = 1 pairs the two halves of
  // an FP32 pair (scalar), the others whole pairs
#pragma unroll
  for (int i = 0; i < E; i += 2) {
    const float p = x[i], q = x[i + 1];
    x[i] = __fadd_rn(p, q);
    x[i + 1] = __fsub_rn(p, q);
  }
#pragma unroll
  for (int len = 2; len < E; len <<= 1) {
#pragma unroll
    for (int i = 0; i < E; i += 2)
      if ((i & len) == 0) butterfly2(x, i, i + len);
  }

  // the transpose: y[4 i + e] = element e of chunk NC rl + (i % NC + rw) % NC
  // of block i / NC
  const uint32_t rbase = smem_u32(&s_rows[warp][0]) + rw * D * 4;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(rbase + rl * 128 + 16 * (c ^ (lane & 7))),
                 "f"(x[4 * c]), "f"(x[4 * c + 1]), "f"(x[4 * c + 2]), "f"(x[4 * c + 3])
                 : "memory");
  }
  __syncwarp();
  float y[E];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int hb = i / NC, j = (i % NC + rw) % NC;
    const uint32_t addr = rbase + hb * 128 + 16 * ((NC * rl + j) ^ ((rw * LPR + hb) & 7));
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(y[4 * i]), "=f"(y[4 * i + 1]), "=f"(y[4 * i + 2]), "=f"(y[4 * i + 3])
                 : "r"(addr)
                 : "memory");
  }
  // stages len = 32 .. D/2: block bit `bit` (slots of block hb at 4 NC hb)
#pragma unroll
  for (int bit = 1; bit < LPR; bit <<= 1) {
#pragma unroll
    for (int hb = 0; hb < LPR; ++hb) {
      if (hb & bit) continue;
#pragma unroll
      for (int e = 0; e < 4 * NC; e += 2) butterfly2(y, 4 * NC * hb + e, 4 * NC * (hb + bit) + e);
    }
  }
  // the scale, negated: y holds -RN(y / sqrt D) (RN is odd), the dividends
  // of div_rn_pair_neg
  {
    const uint64_t sc = f2(-inv_sqrt_d<D>(), -inv_sqrt_d<D>());
#pragma unroll
    for (int i = 0; i < E; i += 2) f2_split(mul_f2(f2(y[i], y[i + 1]), sc), y[i], y[i + 1]);
  }

  // quotients of the rotated values by s as the IEEE division gives them:
  // Markstein's correction step on FP32 pairs where the operands allow it
  // (div_rn_in_range), else the IEEE division
  float lam = 0.f;                                        // the lane's largest |y|
#pragma unroll
  for (int i = 0; i < E; ++i) lam = fmaxf(lam, fabsf(y[i]));
  auto quotients4 = [&](float s, float r, bool in_range, int i0, float (&q)[4]) {
    if (in_range) {
      const uint64_t bb = f2(s, s), ny2 = f2(-r, -r);
      div_rn_pair_neg(y[i0], y[i0 + 1], bb, ny2, q[0], q[1]);
      div_rn_pair_neg(y[i0 + 2], y[i0 + 3], bb, ny2, q[2], q[3]);
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) q[e] = __fdiv_rn(-y[i0 + e], s);
    }
  };
  // element index (in the row) of y[4 i]
  auto elem = [&](int i) { return 32 * (i / NC) + NL * rl + 4 * ((i % NC + rw) % NC); };

  // V: the row's amax over its LPR lanes (before any lane leaves)
  float amax = lam;
#pragma unroll
  for (int o = 1; o < LPR; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));

  if (!live || slot < 0) return;
  const int64_t cap = static_cast<int64_t>(a.num_pages) * a.P;
  if (slot >= cap) {
    if (rl == 0 && kind == 0) set_error(a.err, KV4_EBOUNDS);
    return;
  }
  // slots are below num_pages * P < 2^31 (the pool check), so 32-bit math
  const uint32_t page = fdiv(static_cast<uint32_t>(slot), a.p_div);
  const int off = static_cast<int>(static_cast<uint32_t>(slot) - page * static_cast<uint32_t>(a.P));
  uint8_t* chunk = a.pool + (static_cast<int64_t>(page) * a.Hkv + h) * a.chunk_bytes;

  if (kind == 0) {
    const float s = __ldg(a.s_k), r = __frcp_rn(s);
    const bool in_range = div_rn_in_range(r, lam);
    uint8_t* dst = chunk + static_cast<int64_t>(off) * D;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float q[4];
      quotients4(s, r, in_range, 4 * i, q);
      *reinterpret_cast<uint32_t*>(dst + elem(i)) = f32x2_to_e4m3x2(q[0], q[1]) | (f32x2_to_e4m3x2(q[2], q[3]) << 16);
    }
  } else {
    const float s = div7(amax);                           // RN(amax / 7)
    // V codes in token-pair rows by 16-bit halves: elements e .. e+3 (e a
    // multiple of 4) of this token at byte e + 2 (off % 2) of pair row off / 2
    uint8_t* codes = chunk + static_cast<int64_t>(a.P) * D + static_cast<int64_t>(off >> 1) * D + 2 * (off & 1);
    // |y / s| <= 7.0000005: rint by the magic addition, no clamp needed
    const float r = s != 0.f ? __frcp_rn(s) : 0.f;
    const bool in_range = s != 0.f && div_rn_in_range(r, lam);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t nib = 0;                                   // element e in nibble e
      if (s != 0.f) {
        float q[4];
        quotients4(s, r, in_range, 4 * i, q);
        nib = int4x4(q);
      }
      *reinterpret_cast<uint16_t*>(codes + elem(i)) = static_cast<uint16_t>(nib);
    }
    if (rl == 0)
      *reinterpret_cast<float*>(chunk + static_cast<int64_t>(a.P) * D + static_cast<int64_t>(a.P) * (D / 2) +
                                4 * off) = s;
  }
}

}  // namespace

cudaError_t launch_k8v4_write(const K8V4WriteArgs& a_in, cudaStream_t st) {
  if (a_in.rows == 0) return cudaSuccess;
  K8V4WriteArgs a = a_in;
  a.hkv_div = make_fastdiv(static_cast<uint32_t>(a.Hkv));
  a.p_div = make_fastdiv(static_cast<uint32_t>(a.P));
  const int64_t rows_per_cta = 8 * (32 / (a.D / 32));   // 8 warps of 32 / (D / 32) rows
  const dim3 grid(static_cast<unsigned>((a.rows + rows_per_cta - 1) / rows_per_cta), 2);
  switch (a.D) {
    case 64: k8v4_write_kernel<64><<<grid, 256, 0, st>>>(a); break;
    case 128: k8v4_write_kernel<128><<<grid, 256, 0, st>>>(a); break;
    default: k8v4_write_kernel<256><<<grid, 256, 0, st>>>(a); break;
  }
  return cudaGetLastError();
}

}  // namespace kv4
