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
// its G <= 8 query heads; its 4 warps take 16-token tiles in turn and run
// both products on the tensor cores (m16n8k16 f16 MMAs, FP32 accumulation;
// keys exact in f16, values as exact INT4 codes with the per-token scale
// carried by the softmax weight, split into f16 hi + lo).  The combine merges
// the chunks' (max, sum, partial output) and applies the inverse rotation.
#include <cstdint>

#include "kv4_device.cuh"
#include "kv4_internal.h"

namespace kv4 {
namespace {

constexpr int kMaxG = 8;          // query heads per kv head the decode supports
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

// INT4 nibbles at bits 0-3 and 16-19 (lo) or 4-7 and 20-23 (hi) of x ->
// f16x2 of the signed codes: (n ^ 8) + 1024 as an f16 bit pattern, minus
// 1032 (for hi, the nibble sits 16 times higher and is scaled down first).
__device__ __forceinline__ uint32_t nib_lo_pair(uint32_t x) {
  const uint32_t h = (x & 0x000F000Fu) ^ 0x64086408u;
  return hfma2(h, 0x3C003C00u, 0xE408E408u);
}
__device__ __forceinline__ uint32_t nib_hi_pair(uint32_t x) {
  const uint32_t h = ((x & 0x00F000F0u) ^ 0x00800080u) | 0x64006400u;
  return hfma2(h, 0x2C002C00u, 0xD480D480u);
}

// Tensor-core partial decode over one token range (chunk) of one request and
// kv head: 4 warps, each taking 16-token tiles in turn with its own online
// softmax state, merged at the end.  m16n8k16 f16 MMAs, FP32 accumulation:
//   S^T (16 tokens x 8 heads) = K (exact f16 from E4M3) q_rot^T (f16 hi + lo);
//   O^T (16 dims x 8 heads)  += V^T (INT4 codes, exact) P'^T, where
//   P' = p * s_v(token) is split into f16 hi + lo parts.
// Lane (grp = lane / 4, tig = lane % 4).  K-step j of S covers dims
// (D/4) tig + 4j .. +3 for lane tig (any fixed assignment of dims to k works
// when q uses the same one), so a lane reads one contiguous D/4-byte segment
// of each key row.  O row r of m-tile mi is dim (D/8) grp + 2 mi + (r >= 8),
// so a lane reads one contiguous D/16-byte segment of each value row.
template <int D>
__global__ void __launch_bounds__(128) k8v4_partial_kernel(const K8V4DecodeArgs a) {
  constexpr int KS = D / 16;                  // k-steps of S, m-tiles of O
  constexpr int KSEG = D / 4;                 // key bytes per lane and token
  constexpr int VSEG = D / 16;                // value bytes per lane and token
  __shared__ float qsh[kMaxG * D];
  __shared__ __align__(16) float obuf[4 * kMaxG * D];
  __shared__ float sm_m[4][kMaxG], sm_l[4][kMaxG];
  // per k-step and lane: q hi b0, b1, lo b0, b1 -- read only inside the token
  // loop, so it shares bytes with obuf, written only after every warp's loop
  uint4* qfrag = reinterpret_cast<uint4*>(obuf);

  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int G = a.G, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int grp = lane >> 2, tig = lane & 3;
  const int L = max(0, min(a.seq_lens[b], a.max_pages * a.P));
  if (tid == 0 && c == 0 && a.seq_lens[b] > a.max_pages * a.P) set_error(a.err, KV4_EBOUNDS);
  const int per = (L + a.nchunks - 1) / a.nchunks;
  const int t_begin = min(L, c * per), t_end = min(L, t_begin + per);

  // rotated queries (FP32), then this lane's B fragments of S: head grp
  for (int p = tid; p < G * D; p += blockDim.x) {
    const int g = p / D, d = p % D;
    qsh[p] = __bfloat162float(a.q[(static_cast<int64_t>(b) * a.Hq + h * G + g) * D + d]);
  }
  fwht_smem<D>(qsh, G, 1.0f);
  // The rotated q is an FP32 result: split it into f16 hi + lo parts (two
  // MMAs per k-step), so the scores keep FP32-level accuracy.  The B
  // fragments go to shared memory (one 16-byte load per k-step later).
  if (warp == 0) {
#pragma unroll
    for (int j = 0; j < KS; ++j) {
      const int d = KSEG * tig + 4 * j;
      const float* qq = qsh + grp * D + d;
      const bool hv = grp < G;
      uint32_t f[4];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const uint32_t hi = hv ? pack_f16x2(qq[2 * e], qq[2 * e + 1]) : 0u;
        const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hi));
        f[e] = hi;
        f[2 + e] = hv ? pack_f16x2(qq[2 * e] - hf.x, qq[2 * e + 1] - hf.y) : 0u;
      }
      qfrag[j * 32 + lane] = make_uint4(f[0], f[1], f[2], f[3]);
    }
  }
  __syncthreads();
  const float qk_scale = a.sm_scale * __ldg(a.s_k) * kLog2e;

  const int32_t* bt = a.block_table + static_cast<int64_t>(b) * a.max_pages;
  auto chunk_of = [&](int t) -> const uint8_t* {
    if (t >= t_end) return nullptr;
    const int32_t page = bt[t / a.P];
    if (page < 0 || page >= a.num_pages) {
      set_error(a.err, KV4_EBOUNDS);
      return nullptr;
    }
    return a.pool + (static_cast<int64_t>(page) * a.Hkv + h) * a.chunk_bytes;
  };
  const int64_t vcode0 = static_cast<int64_t>(a.P) * D;           // value codes region
  const int64_t vsc0 = vcode0 + static_cast<int64_t>(a.P) * (D / 2); // value scales region

  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float o[KS][4];
#pragma unroll
  for (int mi = 0; mi < KS; ++mi) o[mi][0] = o[mi][1] = o[mi][2] = o[mi][3] = 0.f;

  // ---- loads of one tile: key segments of tokens grp, grp+8 (+ their value
  //      scales); value segments of tokens 2tig, 2tig+1, 2tig+8, 2tig+9
  struct Tile {
    uint32_t kw[2][KS];
    uint32_t vw[4][(VSEG + 3) / 4];
    float sv[2];
    bool kval[2];
  };
  auto load_tile = [&](int t0, Tile& T) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int t = t0 + grp + 8 * r;
      const uint8_t* ch = chunk_of(t);
      T.kval[r] = ch != nullptr;
      T.sv[r] = 0.f;
      if (T.kval[r]) {
        const int off = t % a.P;
        const uint4* src = reinterpret_cast<const uint4*>(ch + static_cast<int64_t>(off) * D + KSEG * tig);
#pragma unroll
        for (int u = 0; u < KS / 4; ++u) {
          const uint4 w = __ldg(src + u);
          T.kw[r][4 * u] = w.x; T.kw[r][4 * u + 1] = w.y; T.kw[r][4 * u + 2] = w.z; T.kw[r][4 * u + 3] = w.w;
        }
        T.sv[r] = __ldg(reinterpret_cast<const float*>(ch + vsc0 + 4 * off));
      } else {
#pragma unroll
        for (int j = 0; j < KS; ++j) T.kw[r][j] = 0u;
      }
    }
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      const int t = t0 + 2 * tig + (q4 & 1) + 8 * (q4 >> 1);
      const uint8_t* ch = chunk_of(t);
      const uint8_t* src = ch ? ch + vcode0 + static_cast<int64_t>(t % a.P) * (D / 2) + VSEG * grp : nullptr;
      if constexpr (VSEG == 16) {
        const uint4 w = src ? __ldg(reinterpret_cast<const uint4*>(src)) : make_uint4(0u, 0u, 0u, 0u);
        T.vw[q4][0] = w.x; T.vw[q4][1] = w.y; T.vw[q4][2] = w.z; T.vw[q4][3] = w.w;
      } else if constexpr (VSEG == 8) {
        const uint2 w = src ? __ldg(reinterpret_cast<const uint2*>(src)) : make_uint2(0u, 0u);
        T.vw[q4][0] = w.x; T.vw[q4][1] = w.y;
      } else {
        T.vw[q4][0] = src ? __ldg(reinterpret_cast<const uint32_t*>(src)) : 0u;
      }
    }
  };

  // Tile i+1's loads are issued before tile i's math.
  Tile cur, nxt;
  if (t_begin + 16 * warp < t_end) load_tile(t_begin + 16 * warp, cur);
  for (int t0 = t_begin + 16 * warp; t0 < t_end; t0 += 64) {
    if (t0 + 64 < t_end) load_tile(t0 + 64, nxt);
    const auto& kw = cur.kw;
    const auto& vw = cur.vw;
    const auto& sv = cur.sv;
    const auto& kval = cur.kval;
    // ---- S^T = K q_rot^T; acc: (token grp, heads 2tig, 2tig+1), (token grp+8, ...)
    float sacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < KS; ++j) {
      uint32_t a0, a1, a2, a3;
      e4m3x4_to_f16x2x2(kw[0][j], a0, a2);
      e4m3x4_to_f16x2x2(kw[1][j], a1, a3);
      const uint4 qf = qfrag[j * 32 + lane];
      mma_f16_16816(sacc, a0, a1, a2, a3, qf.x, qf.y);
      mma_f16_16816(sacc, a0, a1, a2, a3, qf.z, qf.w);
    }

    // ---- online softmax (base 2) for heads 2tig + cc
    float x[4], tmx[2];
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) x[2 * r + cc] = kval[r] ? sacc[2 * r + cc] * qk_scale : -INFINITY;
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      tmx[cc] = fmaxf(x[cc], x[2 + cc]);
#pragma unroll
      for (int o2 = 4; o2 < 32; o2 <<= 1) tmx[cc] = fmaxf(tmx[cc], __shfl_xor_sync(0xffffffffu, tmx[cc], o2));
    }
    float mnew[2], corr[2];
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      mnew[cc] = fmaxf(m_run[cc], tmx[cc]);
      corr[cc] = (mnew[cc] == -INFINITY) ? 1.f : fast_exp2(m_run[cc] - mnew[cc]);
      m_run[cc] = mnew[cc];
    }
    uint32_t pb[2], pl[2];
    float psum[2] = {0.f, 0.f};
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      float w[2];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const float p = (x[2 * r + cc] == -INFINITY) ? 0.f : fast_exp2(x[2 * r + cc] - mnew[cc]);
        psum[cc] += p;
        w[cc] = kval[r] ? p * sv[r] : 0.f;      // the token's value scale rides on its weight
      }
      const uint32_t hi = pack_f16x2(w[0], w[1]);
      const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hi));
      const uint32_t lo = pack_f16x2(w[0] - hf.x, w[1] - hf.y);
      pb[r] = movmatrix_trans(hi);            // (tokens 2tig, 2tig+1 [+8r]) of head grp
      pl[r] = movmatrix_trans(lo);
    }
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) l_run[cc] = l_run[cc] * corr[cc] + psum[cc];
#pragma unroll
    for (int mi = 0; mi < KS; ++mi) {
      o[mi][0] *= corr[0]; o[mi][1] *= corr[1]; o[mi][2] *= corr[0]; o[mi][3] *= corr[1];
    }

    // ---- O^T += V^T P'^T over m-tiles mi (byte mi of the value segments)
#pragma unroll
    for (int mi = 0; mi < KS; ++mi) {
      const int wj = mi >> 2, mm = mi & 3;
      const uint32_t sel = mm | (mm << 4) | ((4 + mm) << 8) | ((4 + mm) << 12);
      const uint32_t xab = prmt(vw[0][wj], vw[1][wj], sel);
      const uint32_t xcd = prmt(vw[2][wj], vw[3][wj], sel);
      const uint32_t a0 = nib_lo_pair(xab), a1 = nib_hi_pair(xab);
      const uint32_t a2 = nib_lo_pair(xcd), a3 = nib_hi_pair(xcd);
      mma_f16_16816(o[mi], a0, a1, a2, a3, pb[0], pb[1]);
      mma_f16_16816(o[mi], a0, a1, a2, a3, pl[0], pl[1]);
    }
    cur = nxt;
  }

  // ---- merge the 4 warps: row sums over the grp lanes, then in shared memory
#pragma unroll
  for (int cc = 0; cc < 2; ++cc)
#pragma unroll
    for (int o2 = 4; o2 < 32; o2 <<= 1) l_run[cc] += __shfl_xor_sync(0xffffffffu, l_run[cc], o2);
  if (grp == 0) {
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      sm_m[warp][2 * tig + cc] = m_run[cc];
      sm_l[warp][2 * tig + cc] = l_run[cc];
    }
  }
  __syncthreads();
  float f[2];
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {
    const int hd = 2 * tig + cc;
    const float M = fmaxf(fmaxf(sm_m[0][hd], sm_m[1][hd]), fmaxf(sm_m[2][hd], sm_m[3][hd]));
    f[cc] = (m_run[cc] == -INFINITY) ? 0.f : fast_exp2(m_run[cc] - M);
  }
  float* ob = obuf + warp * kMaxG * D;
#pragma unroll
  for (int mi = 0; mi < KS; ++mi) {
    const int d0 = (D / 8) * grp + 2 * mi;
    ob[(2 * tig) * D + d0] = o[mi][0] * f[0];
    ob[(2 * tig + 1) * D + d0] = o[mi][1] * f[1];
    ob[(2 * tig) * D + d0 + 1] = o[mi][2] * f[0];
    ob[(2 * tig + 1) * D + d0 + 1] = o[mi][3] * f[1];
  }
  __syncthreads();
  const int64_t slot = (static_cast<int64_t>(b) * a.Hkv + h) * a.nchunks + c;
  float* wo = a.part_o + slot * kMaxG * D;
  for (int p = tid; p < G * D; p += blockDim.x)
    wo[p] = obuf[p] + obuf[kMaxG * D + p] + obuf[2 * kMaxG * D + p] + obuf[3 * kMaxG * D + p];
  if (tid < G) {
    const float M = fmaxf(fmaxf(sm_m[0][tid], sm_m[1][tid]), fmaxf(sm_m[2][tid], sm_m[3][tid]));
    float Ls = 0.f;
    for (int w = 0; w < 4; ++w)
      if (sm_m[w][tid] != -INFINITY) Ls += sm_l[w][tid] * fast_exp2(sm_m[w][tid] - M);
    a.part_ml[(slot * kMaxG + tid) * 2] = M;
    a.part_ml[(slot * kMaxG + tid) * 2 + 1] = Ls;
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
  k8v4_partial_kernel<D><<<dim3(a.nchunks, a.Hkv, a.B), 128, 0, st>>>(a);
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
