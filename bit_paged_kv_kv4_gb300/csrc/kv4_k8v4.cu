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
// match the test oracle's.
// Chunk of P tokens: [K codes P*D][V codes P*D/2][V scales FP32 * P].
//
// Decode runs the NVFP4 / INT4 decode kernel (kv4_decode4.cu) with FP8 keys:
// q is rotated the same way (q_rot . k_rot = q . k), the softmax runs over
// the dequantised rotated keys, and the combine rotates the merged output
// back (H H = I).
#include <cstdint>

#include "kv4_device.cuh"
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
  const int64_t t = row / a.Hkv;
  const int h = static_cast<int>(row - t * a.Hkv);

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
  const int64_t page = slot / a.P;
  const int off = static_cast<int>(slot - page * a.P);
  uint8_t* chunk = a.pool + (page * a.Hkv + h) * a.chunk_bytes;

  if (kind == 0) {
    const float s = __ldg(a.s_k);
    uint8_t* dst = chunk + static_cast<int64_t>(off) * D + lane * E;
    if constexpr (E == 2) {
      const uint32_t w2 = f32x2_to_e4m3x2(__fdiv_rn(x[0], s), __fdiv_rn(x[1], s));
      *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(w2);
    } else {
      uint32_t w[E / 4];
#pragma unroll
      for (int i = 0; i < E; i += 4)
        w[i / 4] = f32x2_to_e4m3x2(__fdiv_rn(x[i], s), __fdiv_rn(x[i + 1], s)) |
                   (f32x2_to_e4m3x2(__fdiv_rn(x[i + 2], s), __fdiv_rn(x[i + 3], s)) << 16);
      if constexpr (E == 8) *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
      else *reinterpret_cast<uint32_t*>(dst) = w[0];
    }
  } else {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < E; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = __fdiv_rn(amax, 7.0f);
    uint32_t nib = 0;                                     // E nibbles, element 2j low in byte j
    if (s != 0.f) {
#pragma unroll
      for (int i = 0; i < E; ++i) {
        int c = __float2int_rn(__fdiv_rn(x[i], s));
        c = c < -8 ? -8 : (c > 7 ? 7 : c);
        nib |= (static_cast<uint32_t>(c) & 0xFu) << (4 * i);
      }
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

cudaError_t launch_k8v4_write(const K8V4WriteArgs& a, cudaStream_t st) {
  if (a.rows == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>((a.rows + 7) / 8), 2);
  switch (a.D) {
    case 64: k8v4_write_kernel<64><<<grid, 256, 0, st>>>(a); break;
    case 128: k8v4_write_kernel<128><<<grid, 256, 0, st>>>(a); break;
    default: k8v4_write_kernel<256><<<grid, 256, 0, st>>>(a); break;
  }
  return cudaGetLastError();
}

}  // namespace kv4
