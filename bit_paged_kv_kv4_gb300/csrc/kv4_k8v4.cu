// The k8v4 variant ("SGLang's 4-bit KV cache", section "Against what this
// site already established": the other 4-bit KV cache of the month keeps
// keys in FP8 and values in 4 bits and gives both one fixed FP32 Hadamard
// rotation of size D).  H = S_D / sqrt(D) (Sylvester), symmetric and
// orthogonal.
//
// Write (k8v4_write_kernel): one warp per (token, head) row of K or V.  The
// row is rotated in FP32 by the fast Walsh-Hadamard transform, stages
// len = 1, 2, ..., D/2 replacing (x_i, x_{i+len}) by (x_i + x_{i+len},
// x_i - x_{i+len}) (i with bit len clear), then scaled by float32(1/sqrt D);
// a lane holds D/32 consecutive elements, so stages below D/32 stay in the
// lane and the others pair lanes by shuffle.  Keys: E4M3(k_rot / s_K) (one
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
template <int D>
__global__ void __launch_bounds__(256) k8v4_write_kernel(const K8V4WriteArgs a) {
  constexpr int E = D / 32;                               // elements per lane
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int kind = blockIdx.y;                            // 0: K, 1: V
  if (row >= a.rows) return;                              // whole warp
  // rows < 2^31 (host check): 32-bit multiply-high division by Hkv
  const uint32_t t32 = fdiv(static_cast<uint32_t>(row), a.hkv_div);
  const int64_t t = t32;
  const int h = static_cast<int>(static_cast<uint32_t>(row) - t32 * static_cast<uint32_t>(a.Hkv));

  // E consecutive bf16 -> FP32
  const __nv_bfloat16* src = (kind == 0 ? a.k : a.v) + row * D + lane * E;
  float x[E];
#pragma unroll
  for (int i = 0; i < E; i += 2) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(src + i));
    x[i] = f.x;
    x[i + 1] = f.y;
  }
  // FWHT, stages len = 1 .. D/2
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
  for (int ll = 1; ll < 32; ll <<= 1) {                   // len = ll * E
    const bool upper = (lane & ll) != 0;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const float o = __shfl_xor_sync(0xffffffffu, x[i], ll);
      x[i] = upper ? __fsub_rn(o, x[i]) : __fadd_rn(x[i], o);
    }
  }
#pragma unroll
  for (int i = 0; i < E; ++i) x[i] = __fmul_rn(x[i], inv_sqrt_d<D>());

  const int64_t slot = a.slot_mapping[t];
  const int64_t cap = static_cast<int64_t>(a.num_pages) * a.P;
  if (slot < 0) return;
  if (slot >= cap) {
    if (lane == 0 && kind == 0) set_error(a.err, KV4_EBOUNDS);
    return;
  }
  // slots are below num_pages * P < 2^31 (the pool check), so 32-bit math
  const uint32_t page = fdiv(static_cast<uint32_t>(slot), a.p_div);
  const int off = static_cast<int>(static_cast<uint32_t>(slot) - page * static_cast<uint32_t>(a.P));
  uint8_t* chunk = a.pool + (static_cast<int64_t>(page) * a.Hkv + h) * a.chunk_bytes;

  // quotients x / s of the lane's elements as the IEEE division gives them:
  // Markstein's correction step on FP32 pairs where the operands allow it
  // (div_rn_in_range), else the IEEE division
  float lam = 0.f;                                        // the lane's largest |x|
#pragma unroll
  for (int i = 0; i < E; ++i) lam = fmaxf(lam, fabsf(x[i]));
  auto quotients = [&](float s, float (&q)[E]) {
    const float r = __frcp_rn(s);
    if (div_rn_in_range(r, lam)) {
      const uint64_t nb = f2(-s, -s), r2 = f2(r, r);
#pragma unroll
      for (int i = 0; i < E; i += 2) div_rn_pair(x[i], x[i + 1], nb, r2, q[i], q[i + 1]);
    } else {
#pragma unroll
      for (int i = 0; i < E; ++i) q[i] = __fdiv_rn(x[i], s);
    }
  };

  if (kind == 0) {
    float q[E];
    quotients(__ldg(a.s_k), q);
    uint8_t* dst = chunk + static_cast<int64_t>(off) * D + lane * E;
    if constexpr (E == 2) {
      const uint32_t w2 = f32x2_to_e4m3x2(q[0], q[1]);
      *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(w2);
    } else {
      uint32_t w[E / 4];
#pragma unroll
      for (int i = 0; i < E; i += 4)
        w[i / 4] = f32x2_to_e4m3x2(q[i], q[i + 1]) | (f32x2_to_e4m3x2(q[i + 2], q[i + 3]) << 16);
      if constexpr (E == 8) *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
      else *reinterpret_cast<uint32_t*>(dst) = w[0];
    }
  } else {
    float amax = lam;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = div7(amax);                           // RN(amax / 7)
    uint32_t nib = 0;                                     // E nibbles, element 2j low in byte j
    if (s != 0.f) {
      // |x / s| <= 7.0000005: rint by the magic addition, no clamp needed
      float q[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      float qe[E];
      quotients(s, qe);
#pragma unroll
      for (int i = 0; i < E; ++i) q[i] = qe[i];
      nib = int4x8(q);
      if constexpr (E < 8) nib &= (1u << (4 * E)) - 1u;
    }
    uint8_t* codes = chunk + static_cast<int64_t>(a.P) * D + static_cast<int64_t>(off) * (D / 2) + lane * (E / 2);
    if constexpr (E == 8) {
      *reinterpret_cast<uint32_t*>(codes) = nib;
    } else if constexpr (E == 4) {
      *reinterpret_cast<uint16_t*>(codes) = static_cast<uint16_t>(nib);
    } else {
      *codes = static_cast<uint8_t>(nib);
    }
    if (lane == 0)
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
  const dim3 grid(static_cast<unsigned>((a.rows + 7) / 8), 2);
  switch (a.D) {
    case 64: k8v4_write_kernel<64><<<grid, 256, 0, st>>>(a); break;
    case 128: k8v4_write_kernel<128><<<grid, 256, 0, st>>>(a); break;
    default: k8v4_write_kernel<256><<<grid, 256, 0, st>>>(a); break;
  }
  return cudaGetLastError();
}

}  // namespace kv4
