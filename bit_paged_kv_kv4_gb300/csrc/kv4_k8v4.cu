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
// a lane holds 32 consecutive elements, so stages below 32 stay in the lane
// and the others pair the row's lanes by shuffle.  Keys: E4M3(k_rot / s_K) (one
// per-tensor FP32 scale); values: INT4 per row, s = amax / 7,
// code = clamp(rne(v_rot / s), -8, 7).  IEEE FP32 throughout, so the bytes
// match the test oracle's; the divisions take Markstein's correction step
// (the IEEE quotient) and the INT4 codes the round-to-nearest-even magic
// addition, as in kv4_write.cu.
// Chunk of P tokens: [K codes P*D][V codes P*D/2][V scales FP32 * P].
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
// consecutive elements a lane (a warp holds 32 / LPR rows), so stages
// len = 1 .. 16 of the transform stay in the lane and len = 32 .. D/2 pair
// lanes of the row by shuffle.
template <int D>
__global__ void __launch_bounds__(256) k8v4_write_kernel(const K8V4WriteArgs a) {
  constexpr int E = 32;                                   // elements per lane
  constexpr int LPR = D / E;                              // lanes per row
  constexpr int RPW = 32 / LPR;                           // rows per warp
  const int lane = threadIdx.x & 31, rl = lane % LPR;     // the lane's place in its row
  const int64_t row = (static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5)) * RPW + lane / LPR;
  const int kind = blockIdx.y;                            // 0: K, 1: V
  // rows past the end compute on row 0 and store nothing (lanes of a row
  // share the shuffles below, and rows of a warp share the warp)
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
  // FWHT, stages len = 1 .. D/2 in order
#pragma unroll
  for (int len = 1; len < E; len <<= 1) {
#pragma unroll
    for (int i = 0; i < E; ++i) {
      if ((i & len) == 0) {
        const float p = x[i], q = x[i + len];
        x[i] = __fadd_rn(p, q);
        x[i + len] = __fsub_rn(p, q);
      }
    }
  }
#pragma unroll
  for (int ll = 1; ll < LPR; ll <<= 1) {                  // len = ll * E
    // the lower partner keeps x + o, the upper o - x: RN(sgn * x + o) in one
    // fma, sgn = +-1 (sgn * x is exact), the same bits as the add or subtract
    const float sgn = (rl & ll) ? -1.f : 1.f;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const float o = __shfl_xor_sync(0xffffffffu, x[i], ll);
      x[i] = __fmaf_rn(sgn, x[i], o);
    }
  }
#pragma unroll
  for (int i = 0; i < E; ++i) x[i] = __fmul_rn(x[i], inv_sqrt_d<D>());

  // quotients x / s of the lane's elements as the IEEE division gives them:
  // Markstein's correction step on FP32 pairs where the operands allow it
  // (div_rn_in_range), else the IEEE division
  float lam = 0.f;                                        // the lane's largest |x|
#pragma unroll
  for (int i = 0; i < E; ++i) lam = fmaxf(lam, fabsf(x[i]));
  auto quotients8 = [&](float s, float r, bool in_range, int i0, float (&q)[8]) {
    if (in_range) {
      const uint64_t nb = f2(-s, -s), r2 = f2(r, r);
#pragma unroll
      for (int i = 0; i < 8; i += 2) div_rn_pair(x[i0 + i], x[i0 + i + 1], nb, r2, q[i], q[i + 1]);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) q[i] = __fdiv_rn(x[i0 + i], s);
    }
  };

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
    uint4* dst = reinterpret_cast<uint4*>(chunk + static_cast<int64_t>(off) * D + rl * E);
#pragma unroll
    for (int c = 0; c < E / 16; ++c) {
      uint32_t w[4];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float q[8];
        quotients8(s, r, in_range, 16 * c + 8 * hh, q);
        w[2 * hh] = f32x2_to_e4m3x2(q[0], q[1]) | (f32x2_to_e4m3x2(q[2], q[3]) << 16);
        w[2 * hh + 1] = f32x2_to_e4m3x2(q[4], q[5]) | (f32x2_to_e4m3x2(q[6], q[7]) << 16);
      }
      dst[c] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else {
    const float s = div7(amax);                           // RN(amax / 7)
    uint32_t nib[E / 8] = {};                             // element 2j low in byte j
    if (s != 0.f) {
      // |x / s| <= 7.0000005: rint by the magic addition, no clamp needed
      const float r = __frcp_rn(s);
      const bool in_range = div_rn_in_range(r, lam);
#pragma unroll
      for (int c = 0; c < E / 8; ++c) {
        float q[8];
        quotients8(s, r, in_range, 8 * c, q);
        nib[c] = int4x8(q);
      }
    }
    uint8_t* codes = chunk + static_cast<int64_t>(a.P) * D + static_cast<int64_t>(off) * (D / 2) + rl * (E / 2);
    *reinterpret_cast<uint4*>(codes) = make_uint4(nib[0], nib[1], nib[2], nib[3]);
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
