// Paged decode attention over the 4-bit pool, split over the sequence, and
// the log-sum-exp combine of the splits.
//
// "SGLang's 4-bit KV cache", Figure 2: decode "reads NVFP4 directly for native
// FP4 decode with scales"; the page's kernel section describes loading packed
// tiles and E4M3 block scales, unpacking E2M1 with a hardware conversion and
// applying the scales.  INT4 per-token-head follows "KV cache in 4 bits"
// (section "What we changed"): one scale per token and head for K and for V.
//
// Design (GB300, sm_103a):
//  * One CTA = (request b, kv head h, group of <= 8 query heads, split s);
//    4 warps, each streaming its own contiguous run of 64-token tiles.
//  * Each warp keeps a private NS-stage ring in shared memory filled by TMA:
//    the packed code rows of K and V arrive through 2-D tiled loads (16-row
//    boxes, 32/64/128-byte swizzle so the fragment reads are bank-conflict
//    free), the scale rows through 1-D bulk copies; completion is tracked with
//    one mbarrier per stage.  Only lane 0 issues copies; no warp waits on
//    another warp, and every wait is bounded.
//  * Dequantisation happens in registers straight into tensor-core fragments:
//    E2M1 bytes -> f16x2 by the hardware conversion, times the E4M3 block
//    scale (e2m1 * e4m3 is exact in f16); INT4 nibbles -> f16x2 by exponent
//    bias arithmetic, the per-token scale applied to the FP32 scores (K) and
//    to the probabilities (V).
//  * QK^T: A = the query group (16 rows, <= 8 used), B = dequantised K^T,
//    so the score accumulator has exactly the layout PV needs for P^T.
//    PV: A = dequantised V^T (16 head-dim rows), B = P^T.  m16n8k16 f16 MMA,
//    FP32 accumulate.  Online softmax in the base-2 domain.
//  * The 4 warps' partial states merge in shared memory in a fixed order
//    (deterministic).  One split writes `out` directly; more splits write
//    (m_x, l, m_y, o) partials that combine_kernel merges.
#include <cstdint>

#include "kv4_device.cuh"
#include "kv4_internal.h"

namespace kv4 {

namespace {

#ifndef KV4_DECODE_TT
#define KV4_DECODE_TT 32
#endif
#ifndef KV4_DECODE_NS
#define KV4_DECODE_NS 3
#endif
#ifndef KV4_DECODE_MINB
#define KV4_DECODE_MINB 2
#endif
constexpr int kTT = KV4_DECODE_TT;     // tokens per tile (per warp and stage)
constexpr int kSub = 16;               // rows per TMA box (sub-tile; never crosses a page)
constexpr int kNW = 4;                 // warps per CTA
constexpr int kNS = KV4_DECODE_NS;     // stages per warp
constexpr int kMinBlocks = KV4_DECODE_MINB;   // CTAs resident per SM (register budget)
constexpr uint32_t kFull = 0xffffffffu;

template <int D, int FMT>
struct Geo {
  static constexpr int RB = D / 2;                             // code bytes per row
  static constexpr int SB = (FMT == KV4_NVFP4) ? D / 16 : 4;   // scale bytes per row
  static constexpr int KB = D / 8;                             // K code bytes per thread per token
  static constexpr int VB = D / 16;                            // V code bytes per thread per token
  static constexpr int MT = D / 16;                            // m-tiles of PV
  static constexpr int STAGE_USED = kTT * (2 * RB + 2 * SB);
  static constexpr int STAGE = (STAGE_USED + 1023) / 1024 * 1024;
  static constexpr int OFF_VC = kTT * RB;
  static constexpr int OFF_KS = 2 * kTT * RB;
  static constexpr int OFF_VS = 2 * kTT * RB + kTT * SB;
  static constexpr int EPI = kNW * 8 * D * 4 + 3 * kNW * 8 * 4;   // epilogue scratch
  static constexpr int RING = kNW * kNS * STAGE;
  static constexpr int SMEM = (RING > EPI ? RING : EPI) + kNW * kNS * 8 + 1024;
};

// Load `N` bytes (N in {4, 8, 16, 32}) of logical row `row`, starting at
// logical column `col` (a multiple of N), of a swizzled code tile.
template <int RB, int N>
__device__ __forceinline__ void load_row_bytes(uint32_t tile, int row, int col, uint32_t* w) {
  if constexpr (N == 32) {
    uint4 a = lds128(tile + swz<RB>(row, col));
    uint4 b = lds128(tile + swz<RB>(row, col + 16));
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
    w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
  } else if constexpr (N == 16) {
    uint4 a = lds128(tile + swz<RB>(row, col));
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
  } else if constexpr (N == 8) {
    uint2 a = lds64(tile + swz<RB>(row, col));
    w[0] = a.x; w[1] = a.y;
  } else {
    w[0] = lds32(tile + swz<RB>(row, col));
  }
}

// Load `N` scale bytes (N in {1, 2, 4}) at byte `off` of a scale tile.
template <int N>
__device__ __forceinline__ uint32_t load_scale_bytes(uint32_t addr) {
  if constexpr (N == 4) return lds32(addr);
  else if constexpr (N == 2) return lds16(addr);
  else return lds8(addr);
}

// INT4 two's-complement nibbles at bits 0-3 and 16-19 of `x` -> f16x2 codes.
__device__ __forceinline__ uint32_t int4_lo_pair(uint32_t x) {
  const uint32_t h = (x & 0x000F000Fu) ^ 0x64086408u;    // 1024 + (n ^ 8)
  return hfma2(h, 0x3C003C00u, 0xE408E408u);              // * 1 - 1032
}
// INT4 nibbles at bits 4-7 and 20-23 of `x` -> f16x2 codes.
__device__ __forceinline__ uint32_t int4_hi_pair(uint32_t x) {
  const uint32_t h = ((x & 0x00F000F0u) ^ 0x00800080u) | 0x64006400u;  // 1024 + 16 (n ^ 8)
  return hfma2(h, 0x2C002C00u, 0xD480D480u);              // / 16 - 72
}

__device__ __forceinline__ void store_out4(void* out, int out_f32, int64_t idx, float4 r) {
  if (out_f32) {
    *reinterpret_cast<float4*>(static_cast<float*>(out) + idx) = r;
  } else {
    __nv_bfloat162 lo = __floats2bfloat162_rn(r.x, r.y), hi = __floats2bfloat162_rn(r.z, r.w);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&lo);
    pk.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + idx) = pk;
  }
}

}  // namespace

template <int D, int FMT>
__global__ void __launch_bounds__(kNW * 32, kMinBlocks)
decode_split_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tmap) {
  using Gm = Geo<D, FMT>;
  constexpr int RB = Gm::RB, SB = Gm::SB, KB = Gm::KB, VB = Gm::VB, MT = Gm::MT;
  constexpr int NM = kTT / 16;            // 16-token groups per tile (QK m-tiles = PV k-groups)
  extern __shared__ uint8_t smem_raw[];

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int grp = lane >> 2, tig = lane & 3;
  const int split = blockIdx.x, b = blockIdx.z;
  const int ngrp = (a.G + 7) >> 3;
  const int h = blockIdx.y / ngrp;
  const int g0 = (blockIdx.y % ngrp) * 8;
  const int ng = min(8, a.G - g0);
  const int hq0 = h * a.G + g0;
  const int S = a.num_splits;

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t ring = base + warp * kNS * Gm::STAGE;
  const uint32_t bars = base + (Gm::RING > Gm::EPI ? Gm::RING : Gm::EPI) + warp * kNS * 8;

  // ---- sequence range of this CTA and of this warp ------------------------
  int L = a.seq_lens[b];
  const int Lmax = a.max_pages * a.P;
  if (L < 0 || L > Lmax) {
    if (threadIdx.x == 0) set_error(a.err, KV4_EBOUNDS);
    L = L < 0 ? 0 : Lmax;
  }
  const int n_tiles = (L + kTT - 1) / kTT;
  const int per_split = (n_tiles + S - 1) / S;
  const int c_begin = min(n_tiles, split * per_split);
  const int c_end = min(n_tiles, c_begin + per_split);
  const int per_warp = (c_end - c_begin + kNW - 1) / kNW;
  const int w_begin = min(c_end, c_begin + warp * per_warp);
  const int w_end = min(c_end, w_begin + per_warp);
  const int n_my = w_end - w_begin;

  if (lane == 0) {
    for (int s = 0; s < kNS; ++s) mbar_init(bars + 8 * s, 1);
    fence_mbar_init();
  }
  if (threadIdx.x == 0) prefetch_tensormap(&tmap);
  __syncwarp();

  // ---- block-table entries, cached one page index per lane ----------------
  const int32_t* bt = a.block_table + static_cast<int64_t>(b) * a.max_pages;
  const int p_first = (w_begin * kTT) / a.P;
  const int p_last = n_my > 0 ? (min(L, w_end * kTT) - 1) / a.P : p_first - 1;
  auto load_page = [&](int rel) -> int {
    const int pi = p_first + rel;
    return pi <= p_last ? __ldg(bt + pi) : 0;
  };
  int win = 0;
  int pg_cur = load_page(lane);
  int pg_nxt = load_page(32 + lane);
  const uint64_t pol = policy_evict_first();
  const uint8_t* pool = a.pool;

  // Issue the copies of warp-local tile i into stage i % kNS.  Warp-uniform.
  auto issue = [&](int i) {
    const int t0 = (w_begin + i) * kTT;
    const int nsub = min(kTT, L - t0 + kSub - 1) / kSub;     // sub-tiles holding tokens
    const int rel0 = t0 / a.P - p_first;
    while ((rel0 >> 5) > win) {
      ++win;
      pg_cur = pg_nxt;
      pg_nxt = load_page((win + 1) * 32 + lane);
    }
    int pages[kTT / kSub];
#pragma unroll
    for (int u = 0; u < kTT / kSub; ++u) {
      const int rel = (t0 + u * kSub) / a.P - p_first;
      const int pc = __shfl_sync(kFull, pg_cur, rel & 31);
      const int pn = __shfl_sync(kFull, pg_nxt, rel & 31);
      pages[u] = ((rel >> 5) == win) ? pc : pn;
    }
    if (lane == 0) {
      const uint32_t st = ring + (i % kNS) * Gm::STAGE;
      const uint32_t bar = bars + 8 * (i % kNS);
      mbar_arrive_expect_tx(bar, nsub * kSub * (2 * RB + 2 * SB));
#pragma unroll
      for (int u = 0; u < kTT / kSub; ++u) {
        if (u < nsub) {
          int page = pages[u];
          if (page < 0 || page >= a.num_pages) {
            set_error(a.err, KV4_EBOUNDS);
            page = 0;
          }
          const int off = (t0 + u * kSub) % a.P;
          const int64_t chunk = (static_cast<int64_t>(page) * a.Hkv + h) * a.chunk_bytes;
          const int row = static_cast<int>(chunk / RB) + off;
          tma_load_2d(st + u * kSub * RB, &tmap, 0, row, bar, pol);
          tma_load_2d(st + Gm::OFF_VC + u * kSub * RB, &tmap, 0, row + a.P, bar, pol);
          const uint8_t* sc = pool + chunk + static_cast<int64_t>(a.P) * 2 * RB;
          bulk_load(st + Gm::OFF_KS + u * kSub * SB, sc + off * SB, kSub * SB, bar, pol);
          bulk_load(st + Gm::OFF_VS + u * kSub * SB, sc + static_cast<int64_t>(a.P) * SB + off * SB,
                    kSub * SB, bar, pol);
        }
      }
    }
  };

  // ---- query fragments (B operand of S^T = K q^T), f16, power-of-two prescaled
  // Thread (grp, tig) holds query row g0+grp, head-dim range [2*KB*tig, 2*KB*(tig+1)).
  constexpr int QN = 2 * KB;                 // query elements per thread
  float qf[QN];
  {
    const bool row_ok = grp < ng;
    const __nv_bfloat16* qrow = a.q + (static_cast<int64_t>(b) * a.Hq + hq0 + grp) * D + QN * tig;
#pragma unroll
    for (int i = 0; i < QN; i += 8) {
      uint4 v = row_ok ? __ldg(reinterpret_cast<const uint4*>(qrow + i)) : make_uint4(0, 0, 0, 0);
      const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float2 f = __bfloat1622float2(p2[j]);
        qf[i + 2 * j] = f.x;
        qf[i + 2 * j + 1] = f.y;
      }
    }
  }
  float qmax = 0.f;
#pragma unroll
  for (int i = 0; i < QN; ++i) qmax = fmaxf(qmax, fabsf(qf[i]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) qmax = fmaxf(qmax, __shfl_xor_sync(kFull, qmax, o));
  // Keep |q| <= 2^14 in f16 by an exact power of two, undone on the scores.
  float qpre = 1.f;
  if (qmax > 16384.f) {
    int e;
    frexpf(qmax / 16384.f, &e);
    qpre = ldexpf(1.f, -e);
  }
  uint32_t qb[QN / 2];
  if constexpr (FMT == KV4_NVFP4) {
    // k-step kk: k (2tig, 2tig+1) <-> d = base + 4kk + {0,1}; (2tig+8, +9) <-> + {2,3}
#pragma unroll
    for (int i = 0; i < QN / 2; ++i) qb[i] = pack_f16x2(qf[2 * i] * qpre, qf[2 * i + 1] * qpre);
  } else {
    // per 8 elements e: kk even: (e0,e4), (e1,e5); kk odd: (e2,e6), (e3,e7)
#pragma unroll
    for (int j = 0; j < QN / 8; ++j) {
      const float* e = qf + 8 * j;
      qb[4 * j + 0] = pack_f16x2(e[0] * qpre, e[4] * qpre);
      qb[4 * j + 1] = pack_f16x2(e[1] * qpre, e[5] * qpre);
      qb[4 * j + 2] = pack_f16x2(e[2] * qpre, e[6] * qpre);
      qb[4 * j + 3] = pack_f16x2(e[3] * qpre, e[7] * qpre);
    }
  }

  const float gk = (FMT == KV4_NVFP4) ? __ldg(a.gscale) : 1.f;
  const float gv = (FMT == KV4_NVFP4) ? __ldg(a.gscale + 1) : 1.f;
  const float qk_scale = a.sm_scale * gk * 1.4426950408889634f / qpre;   // base-2 logits

  // ---- running softmax state (base 2), for heads g0 + 2tig + c, c = 0, 1 ----
  // m_x: running max of the logits x_t, l_run = sum 2^(x_t - m_x) (partial
  // over this thread's tokens).  The PV weights are w_t = 2^(y_t - m_y) with
  // y_t = x_t (NVFP4) or x_t + log2 s_V(t) (INT4: the per-token V scale rides
  // in the exponent, so every f16 operand stays in [0, 1]);
  // out = 2^(m_y - m_x) * sum_t w_t code_t / l.
  float m_x[2] = {-INFINITY, -INFINITY}, m_y[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  float o[MT][4];
#pragma unroll
  for (int mi = 0; mi < MT; ++mi) o[mi][0] = o[mi][1] = o[mi][2] = o[mi][3] = 0.f;

  int issued = 0;
  for (; issued < kNS && issued < n_my; ++issued) issue(issued);

  bool timed_out = false;
  for (int i = 0; i < n_my; ++i) {
    const uint32_t st = ring + (i % kNS) * Gm::STAGE;
    if (!mbar_wait_bounded(bars + 8 * (i % kNS), (i / kNS) & 1)) {
      // give the copies still in flight a bounded chance to land, then stop
      for (int j = i + 1; j < issued; ++j) mbar_wait_bounded(bars + 8 * (j % kNS), (j / kNS) & 1);
      timed_out = true;
      break;
    }
    const int t0 = (w_begin + i) * kTT;
    const int valid = min(kTT, L - t0);
    const uint32_t sK = st, sV = st + Gm::OFF_VC, sKs = st + Gm::OFF_KS, sVs = st + Gm::OFF_VS;

    // -------- S^T[t][g] = K q^T: NM m-tiles of 16 tokens ----------------------
    // A = dequantised K (rows: tokens 16m+grp and 16m+grp+8), B = q^T.
    // sacc[m]: c0 = (16m+grp, head 2tig), c1 = (16m+grp, 2tig+1),
    //          c2 = (16m+grp+8, 2tig),    c3 = (16m+grp+8, 2tig+1)
    float sacc[NM][4];
    uint32_t kw[NM][2][KB / 4];
#pragma unroll
    for (int m = 0; m < NM; ++m) {
      sacc[m][0] = sacc[m][1] = sacc[m][2] = sacc[m][3] = 0.f;
      load_row_bytes<RB, KB>(sK, 16 * m + grp, KB * tig, kw[m][0]);
      load_row_bytes<RB, KB>(sK, 16 * m + grp + 8, KB * tig, kw[m][1]);
    }
    if constexpr (FMT == KV4_NVFP4) {
      constexpr int NB = D / 64;              // block scales per token this thread needs
      // hs[m][r][j]: f16x2 broadcast of block scale j of token 16m+grp+8r
      uint32_t hs[NM][2][NB < 2 ? 2 : NB];
#pragma unroll
      for (int m = 0; m < NM; ++m) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const uint32_t sc = load_scale_bytes<NB>(sKs + (16 * m + grp + 8 * r) * SB + NB * tig);
#pragma unroll
          for (int j = 0; j < NB; j += 2)   // bytes [s_j s_j s_j+1 s_j+1] -> two broadcasts
            e4m3x4_to_f16x2x2(prmt(sc, 0u, (j == 0) ? 0x1100u : 0x3322u), hs[m][r][j], hs[m][r][j + 1]);
        }
      }
#pragma unroll
      for (int j = 0; j < KB / 4; ++j) {      // word j: k-steps 2j (bytes 0, 1) and 2j+1 (bytes 2, 3)
#pragma unroll
        for (int m = 0; m < NM; ++m) {
          uint32_t c0[4], c1[4];
          e2m1x8_to_f16x2x4(kw[m][0][j], c0);
          e2m1x8_to_f16x2x4(kw[m][1][j], c1);
          const uint32_t s0 = hs[m][0][j >> 1], s1 = hs[m][1][j >> 1];
          mma_f16_16816(sacc[m], hmul2(c0[0], s0), hmul2(c1[0], s1), hmul2(c0[1], s0),
                        hmul2(c1[1], s1), qb[4 * j], qb[4 * j + 1]);
          mma_f16_16816(sacc[m], hmul2(c0[2], s0), hmul2(c1[2], s1), hmul2(c0[3], s0),
                        hmul2(c1[3], s1), qb[4 * j + 2], qb[4 * j + 3]);
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < KB / 4; ++j) {
#pragma unroll
        for (int m = 0; m < NM; ++m) {
          const uint32_t w0 = kw[m][0][j], w1 = kw[m][1][j];
          mma_f16_16816(sacc[m], int4_lo_pair(w0), int4_lo_pair(w1), int4_hi_pair(w0),
                        int4_hi_pair(w1), qb[4 * j + 0], qb[4 * j + 1]);
        }
#pragma unroll
        for (int m = 0; m < NM; ++m) {
          const uint32_t w0 = kw[m][0][j] >> 8, w1 = kw[m][1][j] >> 8;
          mma_f16_16816(sacc[m], int4_lo_pair(w0), int4_lo_pair(w1), int4_hi_pair(w0),
                        int4_hi_pair(w1), qb[4 * j + 2], qb[4 * j + 3]);
        }
      }
    }

    // -------- online softmax (base 2) over this tile ----------------------
    // token of sacc[m][2r + c]: 16m + grp + 8r; head 2tig + c
    float yv[NM][4];                 // INT4: exponent of the PV weight
    float tmx[2] = {-INFINITY, -INFINITY}, tmy[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int m = 0; m < NM; ++m) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int t = 16 * m + grp + 8 * r;
        float sk = 1.f, lsv = 0.f;
        bool vok = true;
        if constexpr (FMT == KV4_INT4_PTH) {
          sk = __uint_as_float(lds32(sKs + 4 * t));
          const float sv = __uint_as_float(lds32(sVs + 4 * t));
          lsv = fast_log2(sv);                // sv == 0: no V weight
          vok = sv > 0.f;
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          float x = sacc[m][2 * r + c] * qk_scale * sk;
          x = (t < valid) ? x : -INFINITY;
          sacc[m][2 * r + c] = x;
          tmx[c] = fmaxf(tmx[c], x);
          if constexpr (FMT == KV4_INT4_PTH) {
            yv[m][2 * r + c] = (t < valid && vok) ? x + lsv : -INFINITY;
            tmy[c] = fmaxf(tmy[c], yv[m][2 * r + c]);
          }
        }
      }
    }
    float corr_x[2], corr_y[2], mx_new[2], my_new[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
#pragma unroll
      for (int o2 = 4; o2 < 32; o2 <<= 1) tmx[c] = fmaxf(tmx[c], __shfl_xor_sync(kFull, tmx[c], o2));
      mx_new[c] = fmaxf(m_x[c], tmx[c]);            // finite: valid >= 1
      corr_x[c] = fast_exp2(m_x[c] - mx_new[c]);     // 0 when m_x == -inf
      m_x[c] = mx_new[c];
      corr_y[c] = corr_x[c];
      my_new[c] = mx_new[c];
      if constexpr (FMT == KV4_INT4_PTH) {
#pragma unroll
        for (int o2 = 4; o2 < 32; o2 <<= 1) tmy[c] = fmaxf(tmy[c], __shfl_xor_sync(kFull, tmy[c], o2));
        my_new[c] = fmaxf(m_y[c], tmy[c]);
        corr_y[c] = (my_new[c] == -INFINITY) ? 1.f : fast_exp2(m_y[c] - my_new[c]);
      }
      m_y[c] = my_new[c];
    }
    // P^T operand of PV per 16-token group m: b0 <- tokens (2tig, 2tig+1) of head grp,
    // b1 <- tokens (8+2tig, 8+2tig+1); transposed from the score layout with movmatrix.
    uint32_t pb[NM][2], pl[NM][2];
    float psum[2] = {0.f, 0.f};
#pragma unroll
    for (int m = 0; m < NM; ++m) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        float w[2];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const float p = fast_exp2(sacc[m][2 * r + c] - mx_new[c]);
          psum[c] += p;
          w[c] = p;
          if constexpr (FMT == KV4_INT4_PTH)
            w[c] = (my_new[c] == -INFINITY) ? 0.f : fast_exp2(yv[m][2 * r + c] - my_new[c]);
        }
        const uint32_t hi = pack_f16x2(w[0], w[1]);
        const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hi));
        const uint32_t lo = pack_f16x2(w[0] - hf.x, w[1] - hf.y);
        pb[m][r] = movmatrix_trans(hi);
        pl[m][r] = movmatrix_trans(lo);
      }
    }
#pragma unroll
    for (int c = 0; c < 2; ++c) l_run[c] = l_run[c] * corr_x[c] + psum[c];
    if (__any_sync(kFull, corr_y[0] != 1.f || corr_y[1] != 1.f)) {
#pragma unroll
      for (int mi = 0; mi < MT; ++mi) {
        o[mi][0] *= corr_y[0]; o[mi][1] *= corr_y[1]; o[mi][2] *= corr_y[0]; o[mi][3] *= corr_y[1];
      }
    }

    // -------- O^T += V^T P^T: NM k-groups of 16 tokens -------------------------
#pragma unroll
    for (int kg = 0; kg < NM; ++kg) {
      const int ta = kg * 16 + 2 * tig;       // tokens ta, ta+1 (k 2tig..) and ta+8, ta+9
      uint32_t wa[VB / 4], wb[VB / 4], wc[VB / 4], wd[VB / 4];
      load_row_bytes<RB, VB>(sV, ta, VB * grp, wa);
      load_row_bytes<RB, VB>(sV, ta + 1, VB * grp, wb);
      load_row_bytes<RB, VB>(sV, ta + 8, VB * grp, wc);
      load_row_bytes<RB, VB>(sV, ta + 9, VB * grp, wd);
      if constexpr (FMT == KV4_NVFP4) {
        // block scales of the thread's head-dim range, per token
        constexpr int NVB = (VB >= 8) ? VB / 8 : 1;
        const int blk0 = (VB * grp) / 8;
        const uint32_t xa = load_scale_bytes<NVB>(sVs + ta * SB + blk0);
        const uint32_t xb = load_scale_bytes<NVB>(sVs + (ta + 1) * SB + blk0);
        const uint32_t xc = load_scale_bytes<NVB>(sVs + (ta + 8) * SB + blk0);
        const uint32_t xd = load_scale_bytes<NVB>(sVs + (ta + 9) * SB + blk0);
        // mask tokens past the end: a zero scale zeroes the (finite) codes
        const uint32_t ma = (ta < valid) ? 0xFFFFu : 0u, mb = (ta + 1 < valid) ? 0xFFFF0000u : 0u;
        const uint32_t mc = (ta + 8 < valid) ? 0xFFFFu : 0u, md = (ta + 9 < valid) ? 0xFFFF0000u : 0u;
        uint32_t sab[2], scd[2];
        {
          // each token's NVB scale bytes -> f16 (one conversion per token pair of bytes)
          uint32_t fa, fb, fc, fd;
          e4m3x4_to_f16x2x2(xa | (xb << 16), fa, fb);
          e4m3x4_to_f16x2x2(xc | (xd << 16), fc, fd);
          sab[0] = prmt(fa, fb, 0x5410u) & (ma | mb);   // block 0: (s(ta), s(tb))
          scd[0] = prmt(fc, fd, 0x5410u) & (mc | md);
          sab[1] = prmt(fa, fb, 0x7632u) & (ma | mb);   // block 1 (NVB == 2)
          scd[1] = prmt(fc, fd, 0x7632u) & (mc | md);
        }
#pragma unroll
        for (int j = 0; j < VB / 4; ++j) {
          const uint32_t lab = (wa[j] & 0x0F0F0F0Fu) | ((wb[j] << 4) & 0xF0F0F0F0u);
          const uint32_t hab = ((wa[j] >> 4) & 0x0F0F0F0Fu) | (wb[j] & 0xF0F0F0F0u);
          const uint32_t lcd = (wc[j] & 0x0F0F0F0Fu) | ((wd[j] << 4) & 0xF0F0F0F0u);
          const uint32_t hcd = ((wc[j] >> 4) & 0x0F0F0F0Fu) | (wd[j] & 0xF0F0F0F0u);
          uint32_t vl[4], vh[4], ul[4], uh[4];
          e2m1x8_to_f16x2x4(lab, vl);
          e2m1x8_to_f16x2x4(hab, vh);
          e2m1x8_to_f16x2x4(lcd, ul);
          e2m1x8_to_f16x2x4(hcd, uh);
#pragma unroll
          for (int mm = 0; mm < 4; ++mm) {
            const int mi = 4 * j + mm;
            const int bj = (VB * grp + mi) / 8 - blk0;
            const uint32_t a0 = hmul2(vl[mm], sab[bj]);
            const uint32_t a1 = hmul2(vh[mm], sab[bj]);
            const uint32_t a2 = hmul2(ul[mm], scd[bj]);
            const uint32_t a3 = hmul2(uh[mm], scd[bj]);
            mma_f16_16816(o[mi], a0, a1, a2, a3, pb[kg][0], pb[kg][1]);
            mma_f16_16816(o[mi], a0, a1, a2, a3, pl[kg][0], pl[kg][1]);
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < VB / 4; ++j) {
#pragma unroll
          for (int mm = 0; mm < 4; ++mm) {
            const int mi = 4 * j + mm;
            const uint32_t sel = mm | (mm << 4) | ((4 + mm) << 8) | ((4 + mm) << 12);
            const uint32_t xab = prmt(wa[j], wb[j], sel);
            const uint32_t xcd = prmt(wc[j], wd[j], sel);
            const uint32_t a0 = int4_lo_pair(xab), a1 = int4_hi_pair(xab);
            const uint32_t a2 = int4_lo_pair(xcd), a3 = int4_hi_pair(xcd);
            mma_f16_16816(o[mi], a0, a1, a2, a3, pb[kg][0], pb[kg][1]);
            mma_f16_16816(o[mi], a0, a1, a2, a3, pl[kg][0], pl[kg][1]);
          }
        }
      }
    }
    __syncwarp();
    if (issued < n_my) issue(issued++);
  }
  if (timed_out && lane == 0) set_error(a.err, KV4_ETIMEOUT);

  // ---- merge the warps' states in shared memory, fixed order --------------
#pragma unroll
  for (int c = 0; c < 2; ++c) {
#pragma unroll
    for (int o2 = 4; o2 < 32; o2 <<= 1) l_run[c] += __shfl_xor_sync(kFull, l_run[c], o2);
  }
  __syncthreads();   // every warp finished reading its ring
  float* sO = reinterpret_cast<float*>(smem_raw + (base - smem_u32(smem_raw)));
  float* sMx = sO + kNW * 8 * D;
  float* sMy = sMx + kNW * 8;
  float* sL = sMy + kNW * 8;
  if (grp == 0) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      sMx[warp * 8 + 2 * tig + c] = m_x[c];
      sMy[warp * 8 + 2 * tig + c] = m_y[c];
      sL[warp * 8 + 2 * tig + c] = l_run[c];
    }
  }
  __syncthreads();
  {
    // this thread's O^T columns: heads 2tig, 2tig+1
    float wgt[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int g = 2 * tig + c;
      float My = -INFINITY;
      for (int w = 0; w < kNW; ++w) My = fmaxf(My, sMy[w * 8 + g]);
      const float mw = sMy[warp * 8 + g];
      wgt[c] = (mw == -INFINITY) ? 0.f : fast_exp2(mw - My);
    }
    float* dst = sO + warp * 8 * D;
#pragma unroll
    for (int mi = 0; mi < MT; ++mi) {
      const int d = 2 * (VB * grp + mi);
      dst[(2 * tig) * D + d] = o[mi][0] * wgt[0];
      dst[(2 * tig + 1) * D + d] = o[mi][1] * wgt[1];
      dst[(2 * tig) * D + d + 1] = o[mi][2] * wgt[0];
      dst[(2 * tig + 1) * D + d + 1] = o[mi][3] * wgt[1];
    }
  }
  __syncthreads();
  for (int e = threadIdx.x * 4; e < ng * D; e += kNW * 32 * 4) {
    const int g = e / D, d = e % D;
    float Mx = -INFINITY, My = -INFINITY;
    for (int w = 0; w < kNW; ++w) {
      Mx = fmaxf(Mx, sMx[w * 8 + g]);
      My = fmaxf(My, sMy[w * 8 + g]);
    }
    float l = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int w = 0; w < kNW; ++w) {
      const float mw = sMx[w * 8 + g];
      l += (mw == -INFINITY) ? 0.f : sL[w * 8 + g] * fast_exp2(mw - Mx);
      const float4 v = *reinterpret_cast<const float4*>(sO + (w * 8 + g) * D + d);
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    const int64_t row = static_cast<int64_t>(b) * a.Hq + hq0 + g;
    if (S == 1) {
      const float inv = (l > 0.f && My != -INFINITY) ? gv * fast_exp2(My - Mx) / l : 0.f;
      float4 r = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
      store_out4(a.out, a.out_f32, row * D + d, r);
    } else {
      const int64_t prow = row * S + split;
      *reinterpret_cast<float4*>(a.part_o + prow * D + d) = acc;
      if (d == 0) *reinterpret_cast<float4*>(a.part_ml + 4 * prow) = make_float4(Mx, l, My, 0.f);
    }
  }
}

// Merge the S split partials (m_x, l, m_y, o) of each (request, query head):
//   Mx = max m_x, My = max m_y, l = sum_s l_s 2^(m_x,s - Mx),
//   out = g_V * 2^(My - Mx) * sum_s o_s 2^(m_y,s - My) / l
// Weights are summed in split order, so the result is deterministic.
__global__ void __launch_bounds__(128)
combine_kernel(const float* __restrict__ part_ml, const float* __restrict__ part_o, int S,
               int D, int Hq, const float* __restrict__ gscale, int use_g, void* out,
               int out_f32) {
  extern __shared__ float sw[];          // [S] weights of o_s
  __shared__ float red[2][4];
  __shared__ float bcast[3];
  const int j = blockIdx.x, b = blockIdx.y;
  const int64_t row = static_cast<int64_t>(b) * Hq + j;
  const float4* ml = reinterpret_cast<const float4*>(part_ml) + row * S;
  const float* po = part_o + row * S * D;
  const int tid = threadIdx.x, nt = blockDim.x;

  float Mx = -INFINITY, My = -INFINITY;
  for (int s = tid; s < S; s += nt) {
    const float4 m = ml[s];
    Mx = fmaxf(Mx, m.x);
    My = fmaxf(My, m.z);
  }
  for (int o = 16; o > 0; o >>= 1) {
    Mx = fmaxf(Mx, __shfl_xor_sync(kFull, Mx, o));
    My = fmaxf(My, __shfl_xor_sync(kFull, My, o));
  }
  if ((tid & 31) == 0) {
    red[0][tid >> 5] = Mx;
    red[1][tid >> 5] = My;
  }
  __syncthreads();
  if (tid == 0) {
    float mx = -INFINITY, my = -INFINITY;
    for (int w = 0; w < (nt + 31) / 32; ++w) {
      mx = fmaxf(mx, red[0][w]);
      my = fmaxf(my, red[1][w]);
    }
    bcast[0] = mx;
    bcast[1] = my;
  }
  __syncthreads();
  Mx = bcast[0];
  My = bcast[1];
  for (int s = tid; s < S; s += nt) {
    const float m = ml[s].z;
    sw[s] = (m == -INFINITY) ? 0.f : fast_exp2(m - My);
  }
  __syncthreads();
  if (tid == 0) {
    float l = 0.f;
    for (int s = 0; s < S; ++s) {
      const float4 m = ml[s];
      l += (m.x == -INFINITY) ? 0.f : m.y * fast_exp2(m.x - Mx);
    }
    bcast[2] = l;
  }
  __syncthreads();
  const float l = bcast[2];
  const float g = use_g ? __ldg(gscale + 1) : 1.f;
  const float inv = (l > 0.f && My != -INFINITY) ? g * fast_exp2(My - Mx) / l : 0.f;
  for (int d = tid * 4; d < D; d += nt * 4) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < S; ++s) {
      const float w = sw[s];
      const float4 v = __ldg(reinterpret_cast<const float4*>(po + static_cast<int64_t>(s) * D + d));
      acc.x += w * v.x; acc.y += w * v.y; acc.z += w * v.z; acc.w += w * v.w;
    }
    store_out4(out, out_f32, row * D + d, make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
  }
}

// ------------------------------------------------------------------ launch
template <int D, int FMT>
static cudaError_t launch_split(const DecodeArgs& a, const CUtensorMap& map, cudaStream_t st) {
  using Gm = Geo<D, FMT>;
  auto* k = decode_split_kernel<D, FMT>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Gm::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int ngrp = (a.G + 7) / 8;
  dim3 grid(a.num_splits, a.Hkv * ngrp, a.B);
  k<<<grid, kNW * 32, Gm::SMEM, st>>>(a, map);
  return cudaGetLastError();
}

int decode_tile_tokens() { return kTT; }
int decode_box_rows() { return kSub; }

cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& map, cudaStream_t st) {
  cudaError_t e;
  if (a.fmt == KV4_NVFP4) {
    switch (a.D) {
      case 64: e = launch_split<64, KV4_NVFP4>(a, map, st); break;
      case 128: e = launch_split<128, KV4_NVFP4>(a, map, st); break;
      default: e = launch_split<256, KV4_NVFP4>(a, map, st); break;
    }
  } else {
    switch (a.D) {
      case 64: e = launch_split<64, KV4_INT4_PTH>(a, map, st); break;
      case 128: e = launch_split<128, KV4_INT4_PTH>(a, map, st); break;
      default: e = launch_split<256, KV4_INT4_PTH>(a, map, st); break;
    }
  }
  if (e != cudaSuccess || a.num_splits == 1) return e;
  const int S = a.num_splits;
  combine_kernel<<<dim3(a.Hq, a.B), 64, S * sizeof(float), st>>>(
      a.part_ml, a.part_o, S, a.D, a.Hq, a.gscale, a.fmt == KV4_NVFP4 ? 1 : 0, a.out, a.out_f32);
  return cudaGetLastError();
}

}  // namespace kv4
