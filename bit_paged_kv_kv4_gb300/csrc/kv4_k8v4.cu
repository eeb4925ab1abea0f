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
// Decode (k8v4_partial_kernel + k8v4_combine_kernel): q is rotated the same
// way (q_rot . k_rot = q . k), the softmax runs over the dequantised rotated
// keys, and the combined output is rotated back (H H = I).  A CTA owns one
// contiguous range (chunk) of one request's tokens and one kv head with all
// its G <= 8 query heads; per sub-block of 256 tokens each thread scores one
// token against the G rotated queries (its whole key row loaded at once) while
// an asynchronous copy brings that token's value row and scale into shared
// memory; then each warp accumulates P V from shared memory over a stride of
// tokens with eight value dimensions per lane.  The combine merges
// the chunks' (max, sum, partial output) and applies the inverse rotation.
#include <algorithm>
#include <cstdint>

#include "kv4_device.cuh"
#include "kv4_internal.h"

namespace kv4 {
namespace {

constexpr int kMaxG = 8;          // query heads per kv head the decode supports
constexpr int kTB = 256;          // tokens per sub-block (= threads per CTA)
constexpr float kLog2e = 1.4426950408889634f;

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

// ---------------------------------------------------------------- decode
// In-place FP32 FWHT of n_vec vectors of length D in shared memory (all
// threads of the block), then scaled by float32(1/sqrt D) * mul.
template <int D>
__device__ void fwht_smem(float* v, int n_vec, float mul) {
  for (int len = 1; len < D; len <<= 1) {
    __syncthreads();
    for (int p = threadIdx.x; p < n_vec * (D / 2); p += blockDim.x) {
      const int vec = p / (D / 2), r = p % (D / 2);
      const int i = (r / len) * 2 * len + (r % len);       // bit len of i clear
      float* b = v + vec * D;
      const float x = b[i], y = b[i + len];
      b[i] = __fadd_rn(x, y);
      b[i + len] = __fsub_rn(x, y);
    }
  }
  __syncthreads();
  for (int p = threadIdx.x; p < n_vec * D; p += blockDim.x) v[p] = v[p] * inv_sqrt_d<D>() * mul;
  __syncthreads();
}

template <int D>
__global__ void __launch_bounds__(kTB, 2) k8v4_partial_kernel(const K8V4DecodeArgs a) {
  constexpr int TPR = D / 8;                  // lanes per value row (8 dims each)
  constexpr int NTG = kTB / TPR;              // token groups in pass 2
  __shared__ float qs[kMaxG * D];             // rotated, pre-scaled queries
  __shared__ float ps[kTB * kMaxG];           // scores, then weights, of the sub-block
  __shared__ float red[kMaxG][kTB / 32];
  __shared__ float mrun[kMaxG], lrun[kMaxG], alpha_s[kMaxG];
  // dynamic: the sub-block's value codes [kTB][D/2] and row scales [kTB]
  // during the token loop; the token groups' partial outputs [NTG][G][D]
  // after it (the same bytes)
  extern __shared__ __align__(16) float dyn_smem[];
  uint8_t* vrow = reinterpret_cast<uint8_t*>(dyn_smem);
  float* vsc = reinterpret_cast<float*>(vrow + kTB * (D / 2));
  float* oacc = dyn_smem;

  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int G = a.G, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int L = max(0, min(a.seq_lens[b], a.max_pages * a.P));
  if (tid == 0 && a.seq_lens[b] > a.max_pages * a.P) set_error(a.err, KV4_EBOUNDS);
  const int per = (L + a.nchunks - 1) / a.nchunks;
  const int t_begin = min(L, c * per), t_end = min(L, t_begin + per);

  // rotated queries, scaled so scores come out in log2 units
  for (int p = tid; p < G * D; p += kTB) {
    const int g = p / D, d = p % D;
    qs[p] = __bfloat162float(a.q[(static_cast<int64_t>(b) * a.Hq + h * G + g) * D + d]);
  }
  fwht_smem<D>(qs, G, a.sm_scale * __ldg(a.s_k) * kLog2e);
  if (tid < kMaxG) { mrun[tid] = -INFINITY; lrun[tid] = 0.f; }

  const int tg = tid / TPR, dg = tid % TPR;   // pass 2: token group, 8-dim group
  float o[kMaxG][8];
#pragma unroll
  for (int g = 0; g < kMaxG; ++g)
#pragma unroll
    for (int k = 0; k < 8; ++k) o[g][k] = 0.f;

  const int32_t* bt = a.block_table + static_cast<int64_t>(b) * a.max_pages;
  auto chunk_of = [&](int t) -> const uint8_t* {
    const int32_t page = bt[t / a.P];
    if (page < 0 || page >= a.num_pages) return nullptr;
    return a.pool + (static_cast<int64_t>(page) * a.Hkv + h) * a.chunk_bytes;
  };

  for (int t0 = t_begin; t0 < t_end; t0 += kTB) {
    // pass 1: thread tid scores token t0 + tid against the G queries and
    // starts the copy of its value row and scale into shared memory
    {
      const int t = t0 + tid;
      float s[kMaxG];
#pragma unroll
      for (int g = 0; g < kMaxG; ++g) s[g] = 0.f;
      bool ok = t < t_end;
      const uint8_t* ch = ok ? chunk_of(t) : nullptr;
      if (ok && ch == nullptr) { set_error(a.err, KV4_EBOUNDS); ok = false; }
      uint8_t* vdst = vrow + tid * (D / 2);
      if (ok) {
        const int off = t % a.P;
        const uint8_t* vsrc = ch + static_cast<int64_t>(a.P) * D + static_cast<int64_t>(off) * (D / 2);
#pragma unroll
        for (int u = 0; u < D / 32; ++u)
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                       :: "r"(smem_u32(vdst + 16 * u)), "l"(vsrc + 16 * u) : "memory");
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;"
                     :: "r"(smem_u32(vsc + tid)),
                        "l"(ch + static_cast<int64_t>(a.P) * D + static_cast<int64_t>(a.P) * (D / 2) + 4 * off)
                     : "memory");
        asm volatile("cp.async.commit_group;" ::: "memory");
        const uint4* krow = reinterpret_cast<const uint4*>(ch + static_cast<int64_t>(off) * D);
        constexpr int KU = D / 16;
        uint4 kw[KU];
#pragma unroll
        for (int u = 0; u < KU; ++u) kw[u] = __ldg(krow + u);     // the whole key row in flight
#pragma unroll
        for (int u = 0; u < KU; ++u) {
          const uint32_t ws[4] = {kw[u].x, kw[u].y, kw[u].z, kw[u].w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint32_t h0, h1;
            e4m3x4_to_f16x2x2(ws[k], h0, h1);
            const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&h0));
            const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&h1));
            const int d = u * 16 + k * 4;
#pragma unroll
            for (int g = 0; g < kMaxG; ++g) {
              if (g < G) {
                const float4 qq = *reinterpret_cast<const float4*>(qs + g * D + d);
                s[g] = fmaf(f0.x, qq.x, fmaf(f0.y, qq.y, fmaf(f1.x, qq.z, fmaf(f1.y, qq.w, s[g]))));
              }
            }
          }
        }
      } else {
#pragma unroll
        for (int u = 0; u < D / 32; ++u) *reinterpret_cast<uint4*>(vdst + 16 * u) = make_uint4(0u, 0u, 0u, 0u);
        vsc[tid] = 0.f;
      }
#pragma unroll
      for (int g = 0; g < kMaxG; ++g) ps[tid * kMaxG + g] = ok ? s[g] : -INFINITY;
      // sub-block maximum per head
#pragma unroll
      for (int g = 0; g < kMaxG; ++g) {
        float m = ok ? s[g] : -INFINITY;
#pragma unroll
        for (int x = 16; x > 0; x >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, x));
        if (lane == 0) red[g][warp] = m;
      }
    }
    __syncthreads();
    if (tid < G) {
      float m = red[tid][0];
      for (int w = 1; w < kTB / 32; ++w) m = fmaxf(m, red[tid][w]);
      const float mn = fmaxf(mrun[tid], m);
      alpha_s[tid] = (mn == -INFINITY) ? 1.f : fast_exp2(mrun[tid] - mn);
      mrun[tid] = mn;
    }
    __syncthreads();
    // weights of this thread's token, and their sum per head
#pragma unroll
    for (int g = 0; g < kMaxG; ++g) {
      float p = 0.f;
      if (g < G) {
        const float sc = ps[tid * kMaxG + g];
        p = (sc == -INFINITY) ? 0.f : fast_exp2(sc - mrun[g]);
        ps[tid * kMaxG + g] = p;
      }
#pragma unroll
      for (int x = 16; x > 0; x >>= 1) p += __shfl_xor_sync(0xffffffffu, p, x);
      if (lane == 0) red[g][warp] = p;
    }
    // rescale the running outputs
#pragma unroll
    for (int g = 0; g < kMaxG; ++g) {
      const float al = (g < G) ? alpha_s[g] : 1.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) o[g][k] *= al;
    }
    asm volatile("cp.async.wait_all;" ::: "memory");      // this thread's value copies
    __syncthreads();
    if (tid < G) {
      float sum = 0.f;
      for (int w = 0; w < kTB / 32; ++w) sum += red[tid][w];
      lrun[tid] = lrun[tid] * alpha_s[tid] + sum;
    }
    // pass 2: token group tg takes tokens t0 + tg, t0 + tg + NTG, ...; lane
    // dg accumulates value dims 8 dg .. 8 dg + 7
    for (int i = tg; i < kTB && t0 + i < t_end; i += NTG) {
      const uint32_t nib = *reinterpret_cast<const uint32_t*>(vrow + i * (D / 2) + 4 * dg);
      const float sv = vsc[i];
      float v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int code = static_cast<int>((nib >> (4 * k)) & 0xFu);
        v[k] = static_cast<float>(code >= 8 ? code - 16 : code) * sv;
      }
#pragma unroll
      for (int g = 0; g < kMaxG; ++g) {
        if (g < G) {
          const float p = ps[i * kMaxG + g];
#pragma unroll
          for (int k = 0; k < 8; ++k) o[g][k] = fmaf(p, v[k], o[g][k]);
        }
      }
    }
    __syncthreads();
  }

  // reduce the token groups' partial outputs and write this chunk's partial
#pragma unroll
  for (int g = 0; g < kMaxG; ++g) {
    if (g < G) {
#pragma unroll
      for (int k = 0; k < 8; ++k) oacc[(tg * G + g) * D + dg * 8 + k] = o[g][k];
    }
  }
  __syncthreads();
  const int64_t slot = (static_cast<int64_t>(b) * a.Hkv + h) * a.nchunks + c;
  float* wo = a.part_o + slot * kMaxG * D;
  for (int p = tid; p < G * D; p += kTB) {
    float sum = 0.f;
    for (int j = 0; j < NTG; ++j) sum += oacc[j * G * D + p];
    wo[p] = sum;
  }
  if (tid < G) {
    a.part_ml[(slot * kMaxG + tid) * 2] = mrun[tid];
    a.part_ml[(slot * kMaxG + tid) * 2 + 1] = lrun[tid];
  }
}

// One CTA per (query head, request): merge the chunks, rotate back, store.
template <int D>
__global__ void __launch_bounds__(D) k8v4_combine_kernel(const K8V4DecodeArgs a) {
  __shared__ float ov[D];
  const int j = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
  const int h = j / a.G, g = j % a.G;
  const int64_t base = (static_cast<int64_t>(b) * a.Hkv + h) * a.nchunks;
  float m = -INFINITY;
  for (int c = 0; c < a.nchunks; ++c) m = fmaxf(m, a.part_ml[((base + c) * kMaxG + g) * 2]);
  float l = 0.f, acc = 0.f;
  if (m != -INFINITY) {
    for (int c = 0; c < a.nchunks; ++c) {
      const float mc = a.part_ml[((base + c) * kMaxG + g) * 2];
      if (mc == -INFINITY) continue;
      const float w = fast_exp2(mc - m);
      l += w * a.part_ml[((base + c) * kMaxG + g) * 2 + 1];
      acc += w * a.part_o[((base + c) * kMaxG + g) * D + d];
    }
  }
  ov[d] = (l > 0.f) ? acc / l : 0.f;
  fwht_smem<D>(ov, 1, 1.0f);
  const int64_t orow = (static_cast<int64_t>(b) * a.Hq + j) * D + d;
  if (a.out_f32) static_cast<float*>(a.out)[orow] = ov[d];
  else static_cast<__nv_bfloat16*>(a.out)[orow] = __float2bfloat16_rn(ov[d]);
}

template <int D>
cudaError_t launch_decode_d(const K8V4DecodeArgs& a, cudaStream_t st) {
  constexpr int NTG = kTB / (D / 8);
  constexpr int kStage = kTB * (D / 2 + 4);
  const size_t dyn = std::max(static_cast<size_t>(NTG) * a.G * D * sizeof(float), static_cast<size_t>(kStage));
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k8v4_partial_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         std::max(NTG * kMaxG * D * static_cast<int>(sizeof(float)), kStage));
    if (e != cudaSuccess) return e;
    attr = true;
  }
  k8v4_partial_kernel<D><<<dim3(a.nchunks, a.Hkv, a.B), kTB, dyn, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  k8v4_combine_kernel<D><<<dim3(a.Hq, a.B), D, 0, st>>>(a);
  return cudaGetLastError();
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

cudaError_t launch_k8v4_decode(const K8V4DecodeArgs& a, cudaStream_t st) {
  switch (a.D) {
    case 64: return launch_decode_d<64>(a, st);
    case 128: return launch_decode_d<128>(a, st);
    default: return launch_decode_d<256>(a, st);
  }
}

}  // namespace kv4
