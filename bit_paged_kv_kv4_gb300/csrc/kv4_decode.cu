// Paged decode attention over the FP8 E4M3 per-tensor pool (the comparison
// format the 4-bit cache is measured against), split over the sequence, and
// the log-sum-exp combine of the pieces, which every format's decode uses
// (the NVFP4, INT4 and k8v4 decode kernel is in kv4_decode4.cu).
//
// Work decomposition (GB300: 152 SMs, two CTAs of 4 warps resident on each):
//  * A unit is (request b, kv head h, slice of <= 8 query heads of h's group);
//    its work is ceil(seq_len / 16) tiles of 16 tokens.  All units' tiles are
//    laid end to end in (b, h, slice, tile) order.
//  * Balanced mode (num_splits != 1): one wave of persistent CTAs; CTA c takes
//    the tiles [c*T/n, (c+1)*T/n) of the whole list, so every CTA streams the
//    same number of bytes whatever the length mix.  Independently, each unit
//    is cut into S equal split ranges (S = num_splits, or 1 when 0 is passed).
//    A piece is the intersection of a CTA range with a split range; it gets
//    workspace slot `c + (u*S + s)`, which is unique because both are ordered
//    partitions of the same line.  combine_kernel merges each unit's pieces.
//    A unit that lies inside one CTA range with S = 1 is written directly.
//  * Unit mode (num_splits == 1): one CTA per unit, output written directly,
//    no workspace.
//  * Inside a CTA, each segment (one piece) is divided among the 4 warps in
//    contiguous runs of tiles; the warps' (m, l, o) states merge in shared
//    memory in warp order (deterministic) at the end of the segment.
//
// Per warp (GB300 data path):
//  * A private 2-stage ring in shared memory filled by TMA: a token's D code
//    bytes are two code rows of D/2, and the K and V rows arrive through 2-D
//    tiled loads (boxes of 16 or 32 rows, 32/64/128-byte swizzle, so the
//    fragment reads are bank-conflict free); one mbarrier per stage, bounded
//    waits.  Block-table entries are prefetched one per lane, 32 pages ahead.
//  * E4M3 -> f16x2 by the hardware conversion straight into tensor-core
//    fragments (exact); the layer's K and V scales act on the scores and on
//    the output.
//  * S^T = K q^T with A = K (16 tokens per MMA) and B = the query slice;
//    movmatrix turns the score tile into the P^T operand of O^T += V^T P^T
//    (A = V^T, 16 head-dim rows per MMA).  m16n8k16 f16 MMA, FP32
//    accumulate; PV weights as f16 hi + lo pairs.
#include <cstdint>
#include <utility>

#include "kv4_device.cuh"
#include "kv4_internal.h"

namespace kv4 {

namespace {

#ifndef KV4_DECODE_NS
#define KV4_DECODE_NS 2
#endif
constexpr int kNW = 4;                 // warps per CTA
constexpr int kNS = KV4_DECODE_NS;     // stages per warp
constexpr int kCtasPerSm = 2;          // resident CTAs per SM (register and smem budget)
constexpr int kMaxSeg = 64;            // segments held in shared memory per pass
constexpr uint32_t kFull = 0xffffffffu;

template <int D, int FMT>
struct Geo {
  static_assert(FMT == KV4_FP8, "the split kernel decodes the FP8 pool");
  static constexpr int TT = 16;                                // tokens per tile
  static constexpr int RPT = 2;                                // code rows per token
  static constexpr int RB = D / 2;                             // code bytes per code row
  static constexpr int SB = 0;                                 // scale bytes per token
  static constexpr int KB = D / 8;                             // K code bytes per thread per token
  static constexpr int VB = D / 16;                            // V code bytes per thread per token
  static constexpr int MT = D / 16;                            // m-tiles of PV
  static constexpr int STAGE_USED = TT * (2 * RPT * RB + 2 * SB);
  static constexpr int STAGE = (STAGE_USED + 1023) / 1024 * 1024;
  static constexpr int OFF_VC = TT * RPT * RB;
  static constexpr int RING = kNW * kNS * STAGE;
  static constexpr int AS = MT * 4 + 4;                        // merge row per lane (floats)
  static constexpr int ACC = 32 * AS * 4;                      // merged O of one segment
  static constexpr int META = kNW * 8 * 3 * 4;                 // (m_x, m_y, l) per warp and head
  static constexpr int SEG = kMaxSeg * 20 + 16;        // keeps the int64 scratch 8-byte aligned
  static constexpr int SMEM = RING + ACC + META + SEG + 64 + kNW * kNS * 8 + 1024;
};

struct Seg {          // one piece: tiles [t0, t0 + n) of unit u, inside split `split`
  int u, t0, n, split, len;   // len: the request's (clamped) sequence length
};

// Load `N` bytes (N in {4, 8, 16, 32}) of a swizzled code row; `a0` is the
// shared address of the first 16-byte unit (or of the N bytes when N < 16),
// `a1` that of the second unit when N == 32.  A TMA swizzle pattern repeats
// every 8 rows, so a thread's addresses are one per-thread constant plus a
// compile-time offset for every row it reads.
template <int N>
__device__ __forceinline__ void load_bytes(uint32_t a0, uint32_t a1, uint32_t* w) {
  if constexpr (N == 32) {
    uint4 x = lds128(a0);
    uint4 y = lds128(a1);
    w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
    w[4] = y.x; w[5] = y.y; w[6] = y.z; w[7] = y.w;
  } else if constexpr (N == 16) {
    uint4 x = lds128(a0);
    w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
  } else if constexpr (N == 8) {
    uint2 x = lds64(a0);
    w[0] = x.x; w[1] = x.y;
  } else {
    w[0] = lds32(a0);
  }
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

// seq_lens[b] clamped to [0, max_pages * P]; a value outside is recorded.
__device__ __forceinline__ int clamp_len(const DecodeArgs& a, int b, bool flag) {
  int L = a.seq_lens[b];
  const int Lmax = a.max_pages * a.P;
  if (L < 0 || L > Lmax) {
    if (flag) set_error(a.err, KV4_EBOUNDS);
    L = L < 0 ? 0 : Lmax;
  }
  return L;
}

// Exclusive prefix of `v` over the CTA's threads; `total` gets the sum.
// `red` is kNW int64 of shared scratch.  Every thread must call it.
__device__ __forceinline__ int64_t block_scan(int64_t v, int64_t* red, int64_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int64_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) red[warp] = x;
  __syncthreads();
  int64_t before = 0;
  total = 0;
#pragma unroll
  for (int w = 0; w < kNW; ++w) {
    const int64_t t = red[w];
    if (w < warp) before += t;
    total += t;
  }
  __syncthreads();
  return before + x - v;
}

}  // namespace

// Partition of [0, total) into `parts` ranges [i*total/parts, (i+1)*total/parts):
// the start of range i, and the range holding x (total > 0, 0 <= x < total).
__host__ __device__ inline int64_t part_begin(int64_t i, int64_t total, int64_t parts) {
  return i * total / parts;
}
__host__ __device__ inline int64_t part_of(int64_t x, int64_t total, int64_t parts) {
  return ((x + 1) * parts - 1) / total;
}

template <int D, int FMT>
__global__ void __launch_bounds__(kNW * 32, kCtasPerSm)
decode_split_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tmap) {
  using Gm = Geo<D, FMT>;
  constexpr int RB = Gm::RB, SB = Gm::SB, KB = Gm::KB, VB = Gm::VB, MT = Gm::MT;
  constexpr int kTT = Gm::TT, RPT = Gm::RPT;
  grid_dep_launch();   // the combine may be scheduled now; it waits for this grid
  grid_dep_wait();     // inputs written by the previous kernel are visible
  constexpr int NM = kTT / 16;            // 16-token groups per tile (QK m-tiles = PV k-groups)
  extern __shared__ uint8_t smem_raw[];

  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int grp = lane >> 2, tig = lane & 3;
  const int ngrp = (a.G + 7) >> 3;
  const int UPB = a.Hkv * ngrp;            // units per request
  const int S = a.num_splits;

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - smem_u32(smem_raw));
  const uint32_t ring = base + warp * kNS * Gm::STAGE;
  float* sAcc = reinterpret_cast<float*>(gbase + Gm::RING);
  float* sMeta = reinterpret_cast<float*>(gbase + Gm::RING + Gm::ACC);
  Seg* sSeg = reinterpret_cast<Seg*>(gbase + Gm::RING + Gm::ACC + Gm::META);
  int64_t* sRed = reinterpret_cast<int64_t*>(gbase + Gm::RING + Gm::ACC + Gm::META + Gm::SEG);
  const uint32_t bars = base + Gm::RING + Gm::ACC + Gm::META + Gm::SEG + 64 + warp * kNS * 8;
  __shared__ int s_nseg;
  __shared__ long long s_cursor, s_cum, s_b;

  if (lane == 0) {
    for (int s2 = 0; s2 < kNS; ++s2) mbar_init(bars + 8 * s2, 1);
    fence_mbar_init();
  }
  if (tid == 0) prefetch_tensormap(&tmap);

  // ---- this CTA's tile range [c0, c1) in the global (b, unit, tile) order ------
  int64_t T = 0, c1 = 0;
  if (a.unit_ctas) {
    // one CTA per unit: the range is that unit's tiles
    const int u = blockIdx.x, b = u / UPB;
    const int n_u = (clamp_len(a, b, tid == 0) + kTT - 1) / kTT;
    if (tid == 0) {
      sSeg[0] = Seg{u, 0, n_u, 0, clamp_len(a, b, false)};
      s_nseg = 1;
    }
  } else {
    for (int b0 = 0; b0 < a.B; b0 += kNW * 32) {
      const int b = b0 + tid;
      const int64_t v = (b < a.B) ? static_cast<int64_t>((clamp_len(a, b, blockIdx.x == 0) + kTT - 1) / kTT) * UPB : 0;
      int64_t tot;
      const int64_t ex = block_scan(v, sRed, tot);
      if (blockIdx.x == 0 && b < a.B) a.cum[b] = T + ex;        // for combine_kernel
      T += tot;
    }
    if (blockIdx.x == 0 && tid == 0) a.cum[a.B] = T;
    c1 = part_begin(blockIdx.x + 1, T, a.n_cta);
    if (tid == 0) s_cursor = part_begin(blockIdx.x, T, a.n_cta);
  }
  __syncthreads();

  // ---- per-thread shared-memory offsets inside a stage ----------------------
  constexpr int D0S = D / 8;                          // V dims (= bytes) per thread
  // FP8: token rows of D bytes (two code rows).  K: thread reads its D/4 bytes
  // of token rows grp (+8); V: its D/8 bytes (dims [D0f, D0f + D/8)) of token
  // rows 2tig, 2tig+1 (+8, +9).  Shifts by multiples of 8 code rows keep the
  // swizzle pattern, so one per-thread constant per row parity suffices.
  const int D0f = D0S * grp;
  const uint32_t k8_off = swz<RB>(2 * grp + (tig >> 1), (D / 4) * (tig & 1));
  const uint32_t k8_off1 = swz<RB>(2 * grp + (tig >> 1), (D / 4) * (tig & 1) + 16);
  const uint32_t k8_off2 = swz<RB>(2 * grp + (tig >> 1), (D / 4) * (tig & 1) + 32);
  const uint32_t k8_off3 = swz<RB>(2 * grp + (tig >> 1), (D / 4) * (tig & 1) + 48);
  const uint32_t v8a0 = Gm::OFF_VC + swz<RB>(4 * tig + D0f / RB, D0f % RB);
  const uint32_t v8a1 = Gm::OFF_VC + swz<RB>(4 * tig + D0f / RB, D0f % RB + 16);
  const uint32_t v8b0 = Gm::OFF_VC + swz<RB>(4 * tig + D0f / RB + 2, D0f % RB);
  const uint32_t v8b1 = Gm::OFF_VC + swz<RB>(4 * tig + D0f / RB + 2, D0f % RB + 16);

  // ---- per-warp running state ----------------------------------------------
  const uint64_t pol = policy_evict_first();
  uint32_t qb[KB];                  // query fragments of the current unit
  float qk_scale = 0.f, gv = 1.f;
  float m_x[2], m_y[2], l_run[2];
  float o[MT][4];
  int issued = 0, consumed = 0;     // warp-local tile counters (stage = counter % kNS)
  bool timed_out = false;

  // passes over the CTA range, kMaxSeg segments at a time
  while (true) {
    if (!a.unit_ctas) {
      // thread 0 lists the next segments of [cursor, c1)
      const int64_t cur = s_cursor;
      __syncthreads();
      if (cur >= c1) break;
      // the request b holding tile `cur` (block scan over b)
      if (tid == 0) s_b = -1;
      __syncthreads();
      int64_t acc = 0;
      for (int b0 = 0; b0 < a.B; b0 += kNW * 32) {
        const int b = b0 + tid;
        const int64_t v = (b < a.B) ? static_cast<int64_t>((clamp_len(a, b, false) + kTT - 1) / kTT) * UPB : 0;
        int64_t tot;
        const int64_t ex = acc + block_scan(v, sRed, tot);
        if (b < a.B && v > 0 && ex <= cur && cur < ex + v) {
          s_b = b;
          s_cum = ex;
        }
        acc += tot;
        __syncthreads();
        if (s_b >= 0) break;
      }
      if (tid == 0) {
        int64_t x = cur;
        int b = static_cast<int>(s_b);
        int64_t cum = s_cum;
        int ns = 0;
        while (x < c1 && ns < kMaxSeg && b >= 0 && b < a.B) {
          const int n_u = (clamp_len(a, b, false) + kTT - 1) / kTT;
          if (n_u == 0 || x >= cum + static_cast<int64_t>(n_u) * UPB) {
            cum += static_cast<int64_t>(n_u) * UPB;
            ++b;
            continue;
          }
          const int64_t rem = x - cum;
          const int j = static_cast<int>(rem / n_u);
          const int t = static_cast<int>(rem % n_u);
          const int split = static_cast<int>(part_of(t, n_u, S));
          const int64_t send = part_begin(split + 1, n_u, S);
          const int n = static_cast<int>(send - t < c1 - x ? send - t : c1 - x);
          sSeg[ns++] = Seg{b * UPB + j, t, n, split, clamp_len(a, b, false)};
          x += n;
        }
        s_nseg = ns;
        s_cursor = (ns == 0) ? c1 : x;     // no segment found: the range is done
      }
      __syncthreads();
    }
    const int nseg = s_nseg;

    // ---- this warp's run of tiles inside segment k ------------------------
    auto my_run = [&](int k, int& beg, int& cnt) {
      const int n = sSeg[k].n;
      const int q = (n + kNW - 1) / kNW;
      beg = min(n, warp * q);
      cnt = min(n, beg + q) - beg;
    };

    // issue cursor and its block-table cache (one page index per lane)
    int ks = -1, io = 0, is_cn = 0, is_bg = 0, is_t0 = 0, is_L = 0, is_h = 0;
    int i_pass = 0, i_total = 0;   // tiles of this pass issued / in total for this warp
    for (int k = 0; k < nseg; ++k) {
      int bg, cn;
      my_run(k, bg, cn);
      i_total += cn;
    }
    int p_first = 0, p_last = -1, win = 0, pg_cur = 0, pg_nxt = 0;
    int pi = 0, po = 0;              // page index and offset of the next tile's first token
    const int32_t* bt = a.block_table;
    const int box = a.box_rows;      // rows per TMA box: 32 when 32 divides P, else 16

    auto issue = [&]() {      // warp-uniform; issues the next tile of this pass
      while (io >= is_cn) {   // enter the next segment with tiles for this warp
        ++ks;
        io = 0;
        my_run(ks, is_bg, is_cn);
        const Seg sg = sSeg[ks];
        const int b = sg.u / UPB;
        is_h = (sg.u % UPB) / ngrp;
        is_t0 = sg.t0;
        is_L = sg.len;
        if (is_cn > 0) {        // reload the page cache for this run
          const int tf = (sg.t0 + is_bg) * kTT;
          pi = tf / a.P;
          po = tf - pi * a.P;
          p_first = pi;
          p_last = (min(is_L, (sg.t0 + is_bg + is_cn) * kTT) - 1) / a.P;
          win = 0;
          bt = a.block_table + static_cast<int64_t>(b) * a.max_pages;
          const int r0 = p_first + lane, r1 = p_first + 32 + lane;
          pg_cur = r0 <= p_last ? __ldg(bt + r0) : 0;
          pg_nxt = r1 <= p_last ? __ldg(bt + r1) : 0;
        }
      }
      const int h = is_h, L = is_L;
      const int t0 = (is_t0 + is_bg + io) * kTT;
      const int boxt = box / RPT;      // tokens per box
      const int nsub = (min(kTT, L - t0) + boxt - 1) / boxt;
      while (((pi - p_first) >> 5) > win) {
        ++win;
        pg_cur = pg_nxt;
        const int r = p_first + (win + 1) * 32 + lane;
        pg_nxt = r <= p_last ? __ldg(bt + r) : 0;
      }
      // the tile's one or two boxes (a box never straddles a page)
      int pu1 = pi, ou1 = po + boxt;
      if (ou1 >= a.P) { ou1 -= a.P; ++pu1; }
      const int rel0 = pi - p_first, rel1 = pu1 - p_first;
      const int pc0 = __shfl_sync(kFull, pg_cur, rel0 & 31), pn0 = __shfl_sync(kFull, pg_nxt, rel0 & 31);
      const int pc1 = __shfl_sync(kFull, pg_cur, rel1 & 31), pn1 = __shfl_sync(kFull, pg_nxt, rel1 & 31);
      const int page0 = ((rel0 >> 5) == win) ? pc0 : pn0;
      const int page1 = ((rel1 >> 5) == win) ? pc1 : pn1;
      if (lane == 0) {
        const uint32_t st = ring + (issued % kNS) * Gm::STAGE;
        const uint32_t bar = bars + 8 * (issued % kNS);
        mbar_arrive_expect_tx(bar, nsub * boxt * (2 * RPT * RB + 2 * SB));
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          if (u < nsub) {
            int page = u ? page1 : page0;
            if (page < 0 || page >= a.num_pages) {
              set_error(a.err, KV4_EBOUNDS);
              page = 0;
            }
            const int off = u ? ou1 : po;
            const int64_t chunk = (static_cast<int64_t>(page) * a.Hkv + h) * a.chunk_bytes;
            const int row = static_cast<int>(chunk / RB) + off * RPT;
            tma_load_2d(st + u * box * RB, &tmap, 0, row, bar, pol);
            tma_load_2d(st + Gm::OFF_VC + u * box * RB, &tmap, 0, row + a.P * RPT, bar, pol);
          }
        }
      }
      po += kTT;                       // advance to the next tile's first token
      while (po >= a.P) { po -= a.P; ++pi; }
      ++io;
      ++issued;
      ++i_pass;
    };

    for (int k0 = 0; k0 < kNS && i_pass < i_total && !timed_out; ++k0) issue();

    for (int k = 0; k < nseg; ++k) {
      const Seg sg = sSeg[k];
      const int b = sg.u / UPB;
      const int h = (sg.u % UPB) / ngrp;
      const int g0 = (sg.u % ngrp) * 8;
      const int ng = min(8, a.G - g0);
      const int hq0 = h * a.G + g0;
      const int L = sg.len;
      int bg, cn;
      my_run(k, bg, cn);

      // ---- query fragments of this unit (B operand of S^T = K q^T) ----------
      // Thread (grp, tig) holds query row g0+grp, head-dim range [2*KB*tig, 2*KB*(tig+1)).
      {
        constexpr int QN = 2 * KB;
        float qf[QN];
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
        float qmax = 0.f;
#pragma unroll
        for (int i = 0; i < QN; ++i) qmax = fmaxf(qmax, fabsf(qf[i]));
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) qmax = fmaxf(qmax, __shfl_xor_sync(kFull, qmax, o2));
        // Keep |q| <= 2^14 in f16 by an exact power of two, undone on the scores.
        float qpre = 1.f;
        if (qmax > 16384.f) {
          int e;
          frexpf(qmax / 16384.f, &e);
          qpre = ldexpf(1.f, -e);
        }
        // k-step kk: k (2tig, 2tig+1) <-> d = base + 4kk + {0,1}; (2tig+8, +9) <-> + {2,3}
#pragma unroll
        for (int i = 0; i < QN / 2; ++i) qb[i] = pack_f16x2(qf[2 * i] * qpre, qf[2 * i + 1] * qpre);
        const float gk = __ldg(a.gscale);
        gv = __ldg(a.gscale + 1);
        qk_scale = a.sm_scale * gk * 1.4426950408889634f / qpre;   // base-2 logits
      }

      // ---- running softmax state (base 2), heads g0 + 2tig + c, c = 0, 1 ------
      // m_x: running max of the logits x_t, l_run = sum 2^(x_t - m_x) (partial
      // over this thread's tokens); the PV weights are w_t = 2^(x_t - m_x) and
      // out = s_V * sum_t w_t code_t / l (m_y = m_x for this format).
      m_x[0] = m_x[1] = m_y[0] = m_y[1] = -INFINITY;
      l_run[0] = l_run[1] = 0.f;
#pragma unroll
      for (int mi = 0; mi < MT; ++mi) o[mi][0] = o[mi][1] = o[mi][2] = o[mi][3] = 0.f;

      for (int jt = 0; jt < cn && !timed_out; ++jt) {
        const uint32_t st = ring + (consumed % kNS) * Gm::STAGE;
        if (!mbar_wait_bounded(bars + 8 * (consumed % kNS), (consumed / kNS) & 1)) {
          // give the copies still in flight a bounded chance to land, then stop
          for (int j = consumed + 1; j < issued; ++j)
            mbar_wait_bounded(bars + 8 * (j % kNS), (j / kNS) & 1);
          timed_out = true;
          break;
        }
        const int t0 = (sg.t0 + bg + jt) * kTT;
        const int valid = min(kTT, L - t0);

        // -------- S^T[t][g] = K q^T: NM m-tiles of 16 tokens ------------------
        // A = dequantised K (rows: tokens 16m+grp and 16m+grp+8), B = q^T.
        // sacc[m]: c0 = (16m+grp, head 2tig), c1 = (16m+grp, 2tig+1),
        //          c2 = (16m+grp+8, 2tig),    c3 = (16m+grp+8, 2tig+1)
        float sacc[NM][4];
#pragma unroll
        for (int m = 0; m < NM; ++m) sacc[m][0] = sacc[m][1] = sacc[m][2] = sacc[m][3] = 0.f;
        {
          // FP8: one E4M3 byte per element; the per-tensor scale is in qk_scale.
          // Word j of a row holds dims 4j..4j+3 of the thread's range = k-step j.
          constexpr int KW8 = D / 16;             // words per row (D/4 bytes)
#pragma unroll
          for (int m = 0; m < NM; ++m) {
            uint32_t k8[2][KW8];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
              const uint32_t rowoff = (32 * m + 16 * r) * RB;      // token rows 16m + 8r (+ grp)
              const uint32_t offs[4] = {k8_off, k8_off1, k8_off2, k8_off3};
#pragma unroll
              for (int u = 0; u < KW8 / 4; ++u) {
                const uint4 x = lds128(st + offs[u] + rowoff);
                k8[r][4 * u] = x.x; k8[r][4 * u + 1] = x.y; k8[r][4 * u + 2] = x.z; k8[r][4 * u + 3] = x.w;
              }
            }
#pragma unroll
            for (int j = 0; j < KW8; ++j) {
              uint32_t a0, a1, a2, a3;
              e4m3x4_to_f16x2x2(k8[0][j], a0, a2);
              e4m3x4_to_f16x2x2(k8[1][j], a1, a3);
              mma_f16_16816(sacc[m], a0, a1, a2, a3, qb[2 * j], qb[2 * j + 1]);
            }
          }
        }

        // -------- online softmax (base 2) over this tile ----------------------
        // token of sacc[m][2r + c]: 16m + grp + 8r; head 2tig + c
        float tmx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int m = 0; m < NM; ++m) {
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int t = 16 * m + grp + 8 * r;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              float x = sacc[m][2 * r + c] * qk_scale;
              x = (t < valid) ? x : -INFINITY;
              sacc[m][2 * r + c] = x;
              tmx[c] = fmaxf(tmx[c], x);
            }
          }
        }
        float corr_x[2], mx_new[2];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
#pragma unroll
          for (int o2 = 4; o2 < 32; o2 <<= 1) tmx[c] = fmaxf(tmx[c], __shfl_xor_sync(kFull, tmx[c], o2));
          mx_new[c] = fmaxf(m_x[c], tmx[c]);            // finite: valid >= 1
          corr_x[c] = fast_exp2(m_x[c] - mx_new[c]);     // 0 when m_x == -inf
          m_x[c] = mx_new[c];
          m_y[c] = mx_new[c];
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
        if (__any_sync(kFull, corr_x[0] != 1.f || corr_x[1] != 1.f)) {
#pragma unroll
          for (int mi = 0; mi < MT; ++mi) {
            o[mi][0] *= corr_x[0]; o[mi][1] *= corr_x[1]; o[mi][2] *= corr_x[0]; o[mi][3] *= corr_x[1];
          }
        }

        // -------- O^T += V^T P^T: NM k-groups of 16 tokens ---------------------
#pragma unroll
        for (int kg = 0; kg < NM; ++kg) {
          const int ta = kg * 16 + 2 * tig;       // tokens ta, ta+1 (k 2tig..) and ta+8, ta+9
          {
            // token rows: word j of each row holds dims D0f + 4j .. +3 of one
            // token; byte-interleave two tokens, then E4M3x2 -> f16x2 gives
            // the (token a, token b) operand registers of two m-tiles
            constexpr int VW8 = D0S / 4;
            uint32_t wa[VW8], wb[VW8], wc[VW8], wd[VW8];
            load_bytes<D0S>(st + v8a0 + 32 * kg * RB, st + v8a1 + 32 * kg * RB, wa);
            load_bytes<D0S>(st + v8b0 + 32 * kg * RB, st + v8b1 + 32 * kg * RB, wb);
            load_bytes<D0S>(st + v8a0 + (32 * kg + 16) * RB, st + v8a1 + (32 * kg + 16) * RB, wc);
            load_bytes<D0S>(st + v8b0 + (32 * kg + 16) * RB, st + v8b1 + (32 * kg + 16) * RB, wd);
            if (valid < kTT) {
              // rows past the end may hold anything, NaN codes included: zero them
#pragma unroll
              for (int j = 0; j < VW8; ++j) {
                wa[j] = (ta < valid) ? wa[j] : 0u;
                wb[j] = (ta + 1 < valid) ? wb[j] : 0u;
                wc[j] = (ta + 8 < valid) ? wc[j] : 0u;
                wd[j] = (ta + 9 < valid) ? wd[j] : 0u;
              }
            }
#pragma unroll
            for (int j = 0; j < VW8; ++j) {
              uint32_t ab0, ab1, ab2, ab3, cd0, cd1, cd2, cd3;
              e4m3x4_to_f16x2x2(prmt(wa[j], wb[j], 0x5140u), ab0, ab1);   // dims +0, +1
              e4m3x4_to_f16x2x2(prmt(wa[j], wb[j], 0x7362u), ab2, ab3);   // dims +2, +3
              e4m3x4_to_f16x2x2(prmt(wc[j], wd[j], 0x5140u), cd0, cd1);
              e4m3x4_to_f16x2x2(prmt(wc[j], wd[j], 0x7362u), cd2, cd3);
              mma_f16_16816(o[2 * j], ab0, ab1, cd0, cd1, pb[kg][0], pb[kg][1]);
              mma_f16_16816(o[2 * j], ab0, ab1, cd0, cd1, pl[kg][0], pl[kg][1]);
              mma_f16_16816(o[2 * j + 1], ab2, ab3, cd2, cd3, pb[kg][0], pb[kg][1]);
              mma_f16_16816(o[2 * j + 1], ab2, ab3, cd2, cd3, pl[kg][0], pl[kg][1]);
            }
          }
        }
        __syncwarp();
        ++consumed;
        if (i_pass < i_total) issue();
      }
      // A warp that timed out stops streaming but still joins every merge below,
      // so the CTA's barriers stay matched; its partial state is empty.


      if (timed_out) {
        m_x[0] = m_x[1] = m_y[0] = m_y[1] = -INFINITY;
        l_run[0] = l_run[1] = 0.f;
#pragma unroll
        for (int mi = 0; mi < MT; ++mi) o[mi][0] = o[mi][1] = o[mi][2] = o[mi][3] = 0.f;
      }
      // ---- merge the warps' states for this segment, in warp order ------------
#pragma unroll
      for (int c = 0; c < 2; ++c) {
#pragma unroll
        for (int o2 = 4; o2 < 32; o2 <<= 1) l_run[c] += __shfl_xor_sync(kFull, l_run[c], o2);
      }
      if (grp == 0) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          float* mt = sMeta + (warp * 8 + 2 * tig + c) * 3;
          mt[0] = m_x[c];
          mt[1] = m_y[c];
          mt[2] = l_run[c];
        }
      }
      __syncthreads();
      float wgt[2];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int g = 2 * tig + c;
        float My = -INFINITY;
        for (int w = 0; w < kNW; ++w) My = fmaxf(My, sMeta[(w * 8 + g) * 3 + 1]);
        const float mw = sMeta[(warp * 8 + g) * 3 + 1];
        wgt[c] = (mw == -INFINITY) ? 0.f : fast_exp2(mw - My);
      }
      // The merge buffer keeps the MMA fragment layout: lane L's o[mi][0..3] at
      // sAcc[L * AS + 4 mi]; the padded row makes every float4 access
      // conflict-free.  Warps add their scaled states in warp order.
      for (int w = 0; w < kNW; ++w) {
        if (warp == w) {
          float* row = sAcc + lane * Gm::AS;
#pragma unroll
          for (int mi = 0; mi < MT; ++mi) {
            float4 v = make_float4(o[mi][0] * wgt[0], o[mi][1] * wgt[1], o[mi][2] * wgt[0], o[mi][3] * wgt[1]);
            if (w != 0) {
              const float4 p = *reinterpret_cast<const float4*>(row + 4 * mi);
              v.x += p.x; v.y += p.y; v.z += p.z; v.w += p.w;
            }
            *reinterpret_cast<float4*>(row + 4 * mi) = v;
          }
        }
        __syncthreads();
      }
      const bool direct = a.unit_ctas || (S == 1 && sg.t0 == 0 && sg.n == (L + kTT - 1) / kTT);
      const int64_t slot = static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(sg.u) * S + sg.split;
      for (int e = tid * 4; e < ng * D; e += kNW * 32 * 4) {
        const int g = e / D, d = e % D;
        float Mx = -INFINITY, My = -INFINITY;
        for (int w = 0; w < kNW; ++w) {
          Mx = fmaxf(Mx, sMeta[(w * 8 + g) * 3 + 0]);
          My = fmaxf(My, sMeta[(w * 8 + g) * 3 + 1]);
        }
        float l = 0.f;
        for (int w = 0; w < kNW; ++w) {
          const float mw = sMeta[(w * 8 + g) * 3 + 0];
          l += (mw == -INFINITY) ? 0.f : sMeta[(w * 8 + g) * 3 + 2] * fast_exp2(mw - Mx);
        }
        // (d, g) lives in lane (grp, tig) with tig = g/2 and grp = the dim chunk
        // q = (d/2) / VB, in o[mi][g%2] with mi = (d/2) % VB; d+1 in
        // o[mi][g%2 + 2]; d+2, d+3 in o[mi+1][...].
        const int hd = d >> 1, mi = hd % VB, c = g & 1;
        const int gq = hd / VB;
        const float* row = sAcc + (gq * 4 + (g >> 1)) * Gm::AS + 4 * mi + c;
        const float4 acc = make_float4(row[0], row[2], row[4], row[6]);
        if (direct) {
          const float inv = (l > 0.f && My != -INFINITY) ? gv * fast_exp2(My - Mx) / l : 0.f;
          const int64_t row = static_cast<int64_t>(b) * a.Hq + hq0 + g;
          store_out4(a.out, a.out_f32, row * D + d,
                     make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
        } else {
          *reinterpret_cast<float4*>(a.part_o + (slot * 8 + g) * D + d) = acc;
          if (d == 0)
            *reinterpret_cast<float4*>(a.part_ml + (slot * 8 + g) * 4) = make_float4(Mx, l, My, 0.f);
        }
      }
      __syncthreads();
    }
    if (a.unit_ctas) break;     // every thread takes the same exit
  }
  if (timed_out && lane == 0) set_error(a.err, KV4_ETIMEOUT);
}

// Merge the pieces of each (request, query head):
//   Mx = max m_x, My = max m_y, l = sum_p l_p 2^(m_x,p - Mx),
//   out = g_V * 2^(My - Mx) * sum_p o_p 2^(m_y,p - My) / l
// The unit's pieces are listed in line order (split by split, CTA by CTA)
// with one thread per split; sums run over fixed thread groups and are
// reduced in a fixed order, so the result is deterministic.
constexpr int kCombineThreads = 256;
constexpr int kMaxPieces = 2048;

// Block-wide max / sum over kCombineThreads threads: a butterfly inside each
// warp, then the warp results in warp order.  The tree is fixed, so a sum is
// the same bits on every run.  `red` holds kCombineThreads / 32 floats.
__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < kCombineThreads / 32; ++w) r = fmaxf(r, red[w]);
  return r;
}
// Two block-wide maxima with one pair of barriers; `red` holds
// 2 * kCombineThreads / 32 floats.
__device__ __forceinline__ void block_max2(float v, float w, float* red, float& rv, float& rw) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    w = fmaxf(w, __shfl_xor_sync(0xffffffffu, w, o));
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) {
    red[threadIdx.x >> 5] = v;
    red[kCombineThreads / 32 + (threadIdx.x >> 5)] = w;
  }
  __syncthreads();
  rv = red[0];
  rw = red[kCombineThreads / 32];
#pragma unroll
  for (int k = 1; k < kCombineThreads / 32; ++k) {
    rv = fmaxf(rv, red[k]);
    rw = fmaxf(rw, red[kCombineThreads / 32 + k]);
  }
}
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < kCombineThreads / 32; ++w) r += red[w];
  return r;
}

__global__ void __launch_bounds__(kCombineThreads)
combine_kernel(const DecodeArgs a) {
  grid_dep_wait();     // the pieces of the split kernel are complete
  __shared__ int64_t s_slot[kMaxPieces];
  __shared__ int64_t s_red[kCombineThreads / 32];
  __shared__ float s_f[2 * kCombineThreads / 32];
  __shared__ float4 s_o[kCombineThreads];
  __shared__ float s_w[kMaxPieces];
  const int j = blockIdx.x, b = blockIdx.y;
  const int D = a.D, S = a.num_splits;
  const int ngrp = (a.G + 7) >> 3, UPB = a.Hkv * ngrp;
  const int h = j / a.G, gi = j % a.G;
  const int u = b * UPB + h * ngrp + gi / 8;
  const int g = gi % 8;
  const int64_t row = static_cast<int64_t>(b) * a.Hq + j;
  int L = a.seq_lens[b];
  const int Lmax = a.max_pages * a.P;
  L = L < 0 ? 0 : (L > Lmax ? Lmax : L);
  const int n_u = (L + a.tile - 1) / a.tile;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  // column block z of gridDim.z: float4 columns [c_lo, c_lo + cols) of the row
  // (k8v4 rotates the whole row, so it runs one block)
  const int cols = D / 4 / static_cast<int>(gridDim.z);
  const int c_lo = static_cast<int>(blockIdx.z) * cols;
  if (n_u == 0) {
    for (int c = tid; c < cols; c += kCombineThreads)
      store_out4(a.out, a.out_f32, row * D + 4 * (c_lo + c), make_float4(0.f, 0.f, 0.f, 0.f));
    return;
  }
  const int64_t T = a.cum[a.B];
  const int64_t start = a.cum[b] + static_cast<int64_t>(u - b * UPB) * n_u;
  if (a.fmt != KV4_K8V4 && S == 1 && part_of(start, T, a.n_cta) == part_of(start + n_u - 1, T, a.n_cta))
    return;  // written directly
  const bool may_be_empty = T < a.n_cta;   // only then can a CTA range hold no tile

  // ---- list the pieces: split s holds CTAs part_of(x0)..part_of(x1-1) ----------
  // One split and no empty CTA range (the usual case): the pieces are the
  // CTAs c0 .. c1 in order, slot c + u.  Otherwise list them in shared memory.
  const int64_t c0 = part_of(start, T, a.n_cta);
  const bool contiguous = (S == 1 && !may_be_empty);
  int64_t npieces = contiguous ? part_of(start + n_u - 1, T, a.n_cta) - c0 + 1 : 0;
  for (int s0 = 0; !contiguous && s0 < S; s0 += kCombineThreads) {
    const int s = s0 + tid;
    int64_t cf = 0, cl = -1;
    if (s < S) {
      const int64_t x0 = start + part_begin(s, n_u, S), x1 = start + part_begin(s + 1, n_u, S);
      if (x1 > x0) {
        cf = part_of(x0, T, a.n_cta);
        cl = part_of(x1 - 1, T, a.n_cta);
      }
    }
    int64_t cnt = 0;
    for (int64_t c = cf; c <= cl; ++c)
      if (!may_be_empty || part_begin(c, T, a.n_cta) != part_begin(c + 1, T, a.n_cta)) ++cnt;
    // exclusive scan of the counts over the block
    int64_t x = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_red[warp] = x;
    __syncthreads();
    int64_t before = 0, tot = 0;
    for (int w = 0; w < kCombineThreads / 32; ++w) {
      if (w < warp) before += s_red[w];
      tot += s_red[w];
    }
    int64_t at = npieces + before + x - cnt;
    for (int64_t c = cf; c <= cl; ++c) {
      if (may_be_empty && part_begin(c, T, a.n_cta) == part_begin(c + 1, T, a.n_cta)) continue;
      if (at < kMaxPieces) s_slot[at] = c + static_cast<int64_t>(u) * S + s;
      ++at;
    }
    npieces += tot;
    __syncthreads();
  }
  const int P = static_cast<int>((contiguous || npieces < kMaxPieces) ? npieces : kMaxPieces);
  if (!contiguous && npieces > kMaxPieces && tid == 0) set_error(a.err, KV4_EUNSUPPORTED);
  auto slot_of = [&](int p) -> int64_t { return contiguous ? c0 + p + u : s_slot[p]; };

  // the thread's first four partial outputs (pieces grp, grp + groups, ...)
  // do not depend on the weights: their loads go out before the reductions
  const int groups = kCombineThreads / cols;     // pieces handled side by side
  const int col = tid % cols, grp = tid / cols;
  const float4* po = reinterpret_cast<const float4*>(a.part_o) + c_lo + col;
  float4 first[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int p = grp + k * groups;
    first[k] = p < P ? __ldg(po + (slot_of(p) * 8 + g) * (D / 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
  }

  // ---- the piece states, read once: maxima, normaliser l, weights ------------
  // Thread t holds pieces t, t + kCombineThreads, ... (at most kPPT of them);
  // each piece's O weight 2^(m_y,p - My) goes to shared memory for the sum.
  constexpr int kPPT = kMaxPieces / kCombineThreads;
  float pmx[kPPT], pl[kPPT], pmy[kPPT];
  float mx = -INFINITY, my = -INFINITY;
#pragma unroll
  for (int k = 0; k < kPPT; ++k) {
    const int p = tid + k * kCombineThreads;
    pmx[k] = pmy[k] = -INFINITY;
    pl[k] = 0.f;
    if (p < P) {
      const float4 m = *reinterpret_cast<const float4*>(a.part_ml + (slot_of(p) * 8 + g) * 4);
      pmx[k] = m.x; pl[k] = m.y; pmy[k] = m.z;
      mx = fmaxf(mx, m.x);
      my = fmaxf(my, m.z);
    }
  }
  float Mx, My;
  block_max2(mx, my, s_f, Mx, My);
  // per-thread partial sums, then a fixed reduction tree: deterministic
  float lp = 0.f;
#pragma unroll
  for (int k = 0; k < kPPT; ++k) {
    const int p = tid + k * kCombineThreads;
    lp += (pmx[k] == -INFINITY) ? 0.f : pl[k] * fast_exp2(pmx[k] - Mx);
    if (p < P) s_w[p] = (pmy[k] == -INFINITY) ? 0.f : fast_exp2(pmy[k] - My);
  }
  const float l = block_sum(lp, s_f);      // its barriers also publish s_w

  // ---- weighted sum of the pieces' o: thread = (piece group, 4 columns) --------
  // pieces grp, grp + groups, ... in that order, four loads in flight at a time
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int p = grp + k * groups;
    if (p < P) {
      const float w = s_w[p];
      acc.x += w * first[k].x; acc.y += w * first[k].y; acc.z += w * first[k].z; acc.w += w * first[k].w;
    }
  }
  int p = grp + 4 * groups;
  for (; p + 3 * groups < P; p += 4 * groups) {
    float4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) v[k] = __ldg(po + (slot_of(p + k * groups) * 8 + g) * (D / 4));
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float w = s_w[p + k * groups];
      acc.x += w * v[k].x; acc.y += w * v[k].y; acc.z += w * v[k].z; acc.w += w * v[k].w;
    }
  }
  for (; p < P; p += groups) {
    const float w = s_w[p];
    const float4 v = __ldg(po + (slot_of(p) * 8 + g) * (D / 4));
    acc.x += w * v.x; acc.y += w * v.y; acc.z += w * v.z; acc.w += w * v.w;
  }
  s_o[tid] = acc;
  __syncthreads();
  float4 res = make_float4(0.f, 0.f, 0.f, 0.f);
  if (grp == 0) {
    for (int r = 1; r < groups; ++r) {
      const float4 v = s_o[r * cols + col];
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    // NVFP4 and FP8 carry the layer's V scale; INT4 and k8v4 put a scale per
    // token into the weights
    const float gv = (a.fmt == KV4_NVFP4 || a.fmt == KV4_FP8) ? __ldg(a.gscale + 1) : 1.f;
    const float inv = (l > 0.f && My != -INFINITY) ? gv * fast_exp2(My - Mx) / l : 0.f;
    res = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  }
  if (a.fmt != KV4_K8V4) {
    if (grp == 0) store_out4(a.out, a.out_f32, row * D + 4 * (c_lo + col), res);
    return;
  }
  // k8v4: the pieces hold sum p V_rot; o = H o_rot with H = S_D / sqrt(D), the
  // Walsh-Hadamard butterflies over the row in FP32
  __shared__ float s_row[kCombineThreads * 4];
  if (grp == 0) *reinterpret_cast<float4*>(s_row + 4 * col) = res;
  for (int len = 1; len < D; len <<= 1) {
    __syncthreads();
    for (int p = tid; p < D / 2; p += kCombineThreads) {
      float* v = s_row + (p / len) * 2 * len + (p % len);
      const float x0 = v[0], x1 = v[len];
      v[0] = __fadd_rn(x0, x1);
      v[len] = __fsub_rn(x0, x1);
    }
  }
  __syncthreads();
  if (grp == 0) {
    const float r = rsqrtf(static_cast<float>(D));
    const float4 v = *reinterpret_cast<const float4*>(s_row + 4 * col);
    store_out4(a.out, a.out_f32, row * D + 4 * col, make_float4(v.x * r, v.y * r, v.z * r, v.w * r));
  }
}

// ------------------------------------------------------------------ launch
// Launch with programmatic stream serialisation: the kernel may be scheduled
// while the previous kernel on the stream drains (its launch latency hides
// behind that kernel's tail); it reads nothing before grid_dep_wait().
template <typename... P, typename... A>
static cudaError_t launch_pdl(void (*k)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              A&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, std::forward<A>(args)...);
}

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
  return launch_pdl(k, dim3(a.n_cta), dim3(kNW * 32), Gm::SMEM, st, a, map);
}

// NVFP4 and INT4 run decode4_kernel (kv4_decode4.cu): 16-token tiles as well.
int decode_tile_tokens(int fmt) { return Geo<256, KV4_FP8>::TT; }

int decode_ctas_per_sm(int fmt) { return fmt == KV4_FP8 ? kCtasPerSm : decode4_ctas_per_sm(); }

int decode_max_ctas_per_sm() { return kCtasPerSm > decode4_ctas_per_sm() ? kCtasPerSm : decode4_ctas_per_sm(); }

cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& map, const CUtensorMap& smap,
                          cudaStream_t st) {
  cudaError_t e;
  if (a.fmt == KV4_FP8) {
    switch (a.D) {
      case 64: e = launch_split<64, KV4_FP8>(a, map, st); break;
      case 128: e = launch_split<128, KV4_FP8>(a, map, st); break;
      default: e = launch_split<256, KV4_FP8>(a, map, st); break;
    }
  } else {
    e = launch_decode4(a, map, smap, st);
  }
  if (e != cudaSuccess || a.unit_ctas) return e;
  // Few output rows (a small batch at long context, each row merging many
  // pieces): split the rows into column blocks of 32 floats or more, up to
  // about two CTAs per SM; many rows: one CTA a row.  (k8v4 rotates whole
  // rows.)
  static int sms[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64) dev = 63;
  if (sms[dev] == 0 && cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms[dev] = 152;
  const int64_t rows = static_cast<int64_t>(a.Hq) * a.B;
  const int64_t want = (2 * static_cast<int64_t>(sms[dev]) + rows - 1) / rows;
  int64_t cz = 1;                               // a power of two that divides D / 32
  while (2 * cz <= want && 2 * cz <= a.D / 32) cz *= 2;
  if (a.fmt == KV4_K8V4) cz = 1;
  return launch_pdl(combine_kernel, dim3(a.Hq, a.B, static_cast<unsigned>(cz)), dim3(kCombineThreads), 0, st, a);
}

}  // namespace kv4
