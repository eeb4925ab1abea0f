// Paged decode attention over the NVFP4 and INT4 pools and the k8v4 pool
// (the FP8 comparison format runs the kernel in kv4_decode.cu).
//
// "SGLang's 4-bit KV cache", Figure 2: decode reads the 4-bit pool as it is
// stored, block scales included, and dequantises inside the kernel; the
// page's kernel section names the hardware E2M1 unpack and the multiply by
// the E4M3 scales.  INT4 per-token-head follows "KV cache in 4 bits", section
// "What we changed": one scale per token and head for K and for V.
//
// Work decomposition: the tile line, balanced CTA ranges, split ranges,
// pieces and their workspace slots are those described in kv4_decode.cu, with
// 16-token tiles (so a tile never straddles a page: P is a multiple of 16),
// and three CTAs of four warps on each SM (at most 168 registers a thread).
// Inside a CTA each segment (one piece) is cut into four runs of consecutive
// tiles, one per warp; at the segment's end the warps' (m, l, O) merge in
// shared memory in warp order (deterministic) and one piece, or the output,
// is written.
//
// Per warp, per tile:
//  * a private ring of NS stages (3) filled by two TMA copies a tile: one 3-D box
//    of the tile's 16 K code rows and 16 V code rows (swizzled so the
//    fragment reads are bank-conflict free) and one of its K and V scale rows,
//    both completing on the stage's mbarrier.  The page of the next tile comes
//    from a block-table cache of one page index per lane; the TMA row and
//    the scale address of a page are computed once per page.
//  * S^T = K q^T on the tensor cores: dequantised K is the A operand (16
//    tokens by 16 dims per m16n8k16 MMA, two accumulation chains), the query
//    slice the B operand, read from a per-CTA copy in shared memory.
//  * an online softmax in base 2 whose base m rises only when a logit
//    exceeds it by more than kLazy, so most tiles need neither a cross-lane
//    maximum nor a rescale of O; the weights (below 2^kLazy) go to the PV MMAs
//    as f16 hi + lo pairs (about 22 significant bits), transposed into the
//    B-operand layout with movmatrix.  INT4's per-token V scale rides on the
//    weight: w = p * s_V(t) / s_ref, s_ref the largest V scale seen so far
//    (raised only when exceeded), and the piece's m_y = m_x + log2(s_ref)
//    carries it to the merge and to the combine kernel.
//  * O^T += V^T P^T with dequantised V^T as the A operand.  V is stored in
//    token pairs: for NVFP4 one hardware E2M1 conversion of a stored byte is
//    one A-fragment register (two tokens of one dim), times the pair's
//    scales; for INT4 and k8v4 (pair rows by 16-bit halves) it is one
//    mask-and-bias conversion of a stored word shifted by 0 or 8 bits.
//
// k8v4 (keys FP8 E4M3 of D bytes a token under one FP32 scale, values INT4
// with a scale per token, both rotated by H = S_D / sqrt(D)) runs the same
// loop: its K box is a 4-D copy of the tile's key rows as lines of at most
// 128 bytes, its V box a 3-D copy of the value pair rows and its 16 V scales one
// 64-byte bulk copy, in two ring stages per warp (a stage is half as large
// again).  The unit's queries are rotated at the segment's start (FP32
// butterflies; the 1/sqrt(D) joins qk_scale) and kept as f16 hi + lo
// fragments, so S^T takes two MMAs per k-step against the exact f16 keys;
// the V scale rides on the weight as for INT4; the output always goes out as
// pieces, and the combine rotates the merged row back.
//
// Every mbarrier wait is bounded (about a second); a warp that runs out
// records KV4_ETIMEOUT, lets its copies in flight land (bounded), stops
// streaming and keeps joining the CTA's barriers, so the CTA drains and exits.
#include <cstdint>
#include <utility>

#include "kv4_device.cuh"
#include "kv4_encode.cuh"
#include "kv4_internal.h"

namespace kv4 {

namespace {

constexpr int kNW = 4;                     // warps per CTA
constexpr int kNS = 3;                     // ring stages per warp
constexpr int kTT = 16;                    // tokens per tile
constexpr int kCtas = 3;                   // resident CTAs per SM
constexpr int kMaxSeg = 64;                // segments listed per pass
constexpr float kLazy = 8.f;
// Code words per row loaded at a time in the K and the NVFP4 V loops
// (shorter live ranges against the 168-register budget of three CTAs).
constexpr int KCW = 4;
constexpr int VCW = 4;
constexpr uint32_t kFull = 0xffffffffu;

template <int D, int FMT>
struct Geo4 {
  static constexpr bool K8 = FMT == KV4_K8V4;                    // FP8 keys, INT4 values, rotated
  static constexpr bool PTV = FMT != KV4_NVFP4;                  // a V scale per token (INT4, k8v4)
  static constexpr int NS = K8 ? 2 : kNS;                        // ring stages per warp
  static constexpr int RB = D / 2;                               // 4-bit code row bytes
  static constexpr int KRB = K8 ? D : RB;                        // K row bytes
  static constexpr int KHB = KRB < 128 ? KRB : 128;              // K line bytes (one swizzle span)
  static constexpr int KH = KRB / KHB;                           // K lines per token
  static constexpr int SB = (FMT == KV4_NVFP4) ? D / 16 : 4;     // scale bytes per token
  static constexpr int KB = K8 ? D / 4 : D / 8;                  // K code bytes per thread per token
  static constexpr int KS = D / 16;                              // k-steps of S (16 dims each)
  static constexpr int VB = D / 16;
  static constexpr int MT = D / 16;                              // m-tiles of PV
  static constexpr int CSK = kTT * KRB;                          // K code bytes of a tile
  static constexpr int CS = kTT * RB;                            // V code bytes of a tile
  static constexpr int STC = CSK + CS;                           // code stage: K box, then V box
  static constexpr int STS = K8 ? kTT * 4 : 2 * kTT * SB;        // scale stage: (K rows), V rows
  static constexpr int VS = K8 ? 0 : kTT * SB;                   // V scales inside the scale stage
  static constexpr int OFF_C = 0;
  static constexpr int OFF_S = OFF_C + kNW * NS * STC;
  static constexpr int OFF_Q = (OFF_S + kNW * NS * STS + 15) / 16 * 16;
  // query fragments: 16 bytes per lane for every k-step (k8v4: q_rot hi + lo)
  // or for every two (one f16 query)
  static constexpr int QF = K8 ? KS * 512 : KB * 128;
  static constexpr int AS = MT * 4 + 4;                          // merge row per lane (floats)
  static constexpr int OFF_ACC = OFF_Q + QF;
  static constexpr int OFF_META = OFF_ACC + 32 * AS * 4;
  static constexpr int OFF_SEG = (OFF_META + kNW * 8 * 3 * 4 + 15) / 16 * 16;
  static constexpr int OFF_RED = OFF_SEG + kMaxSeg * 24;
  static constexpr int OFF_BAR = OFF_RED + kNW * 8;
  static constexpr int SMEM = OFF_BAR + kNW * NS * 8 + 1024;
  // k8v4 rotates the unit's queries in the merge buffer (8 heads x D FP32)
  static_assert(!K8 || 32 * AS * 4 >= 8 * D * 4, "query scratch");
  static_assert(VS >= 0 && KH * KHB == KRB, "stage layout");
};

struct Seg {          // one piece: tiles [t0, t0 + n) of unit u, inside split `split`
  int u, t0, n, split, len;
};

template <int N>
__device__ __forceinline__ void load_bytes(uint32_t a0, uint32_t* w) {
  if constexpr (N == 16) {
    uint4 x = lds128(a0);
    w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
  } else if constexpr (N == 8) {
    uint2 x = lds64(a0);
    w[0] = x.x; w[1] = x.y;
  } else {
    w[0] = lds32(a0);
  }
}

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

__host__ __device__ inline int64_t part_begin4(int64_t i, int64_t total, int64_t parts) {
  return i * total / parts;
}
__host__ __device__ inline int64_t part_of4(int64_t x, int64_t total, int64_t parts) {
  return ((x + 1) * parts - 1) / total;
}

}  // namespace

// ---------------------------------------------------------------- new tokens
// kv4_decode_step: the new token of request b (position L - 1) for kv head h
// goes into the pool before any tile is loaded.  A job is {b, h, page,
// offset in the page} (the page looked up once, by the thread that found
// the job); false when the request is empty or its page is out of range
// (recorded).
__device__ __forceinline__ bool new_token_job(const DecodeArgs& a, int b, int h, int4& job) {
  const int L = clamp_len(a, b, false);
  if (L == 0) return false;
  const int pos = L - 1, pidx = pos / a.P;
  const int page = __ldg(a.block_table + static_cast<int64_t>(b) * a.max_pages + pidx);
  if (page < 0 || page >= a.num_pages) {
    set_error(a.err, KV4_EBOUNDS);
    return false;
  }
  job = make_int4(b, h, page, pos - pidx * a.P);
  return true;
}

// One job's tensor `kind` (0: K, 1: V), quantised by one warp exactly as
// kv4_write does it (the same IEEE FP32 quotients and conversions).  A lane
// holds E = D / 32 consecutive elements; a 16-element NVFP4 block spans
// 16 / E lanes.  Only the CTA that decodes position L - 1 writes it, before
// it loads that tile, so no other thread touches these bytes meanwhile (the
// NVFP4 V pair row is updated by a plain read-modify-write).
template <int D, int FMT>
__device__ __forceinline__ void write_new_token(const DecodeArgs& a, const int4 job, int kind) {
  constexpr int E = D / 32, RB = D / 2;
  const int lane = threadIdx.x & 31;
  const int b = job.x, h = job.y, page = job.z, off = job.w;
  // the pool is written only here, by the one CTA that owns this position
  uint8_t* chunk = const_cast<uint8_t*>(a.pool) + (static_cast<int64_t>(page) * a.Hkv + h) * a.chunk_bytes;
  const __nv_bfloat16* src = (kind == 0 ? a.k_new : a.v_new) + (static_cast<int64_t>(b) * a.Hkv + h) * D + lane * E;
  float x[E];
#pragma unroll
  for (int i = 0; i < E; i += 2) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(src + i));
    x[i] = f.x;
    x[i + 1] = f.y;
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < E; ++i) amax = fmaxf(amax, fabsf(x[i]));
  // q_i = RN(x_i / b) (div_rn on pairs where in range, else IEEE), q = 0 if b = 0
  auto quotients = [&](float bden, float bound, float (&q)[E]) {
    const float yb = __frcp_rn(bden);
    if (div_rn_in_range(yb, bound)) {
      const uint64_t nb = f2(-bden, -bden), yb2 = f2(yb, yb);
#pragma unroll
      for (int i = 0; i < E; i += 2) div_rn_pair(x[i], x[i + 1], nb, yb2, q[i], q[i + 1]);
    } else {
#pragma unroll
      for (int i = 0; i < E; ++i) q[i] = __fdiv_rn(x[i], bden);
    }
  };
  if constexpr (FMT == KV4_NVFP4) {
    constexpr int BL = 16 / E;                            // lanes per block
    constexpr int SB = D / 16;
#pragma unroll
    for (int o = 1; o < BL; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float g = __ldg(a.gscale + kind);
    const float g6 = __fmul_rn(kE2M1Max, g);
    const uint32_t S = f32_to_e4m3(div_rn(amax, g6, __frcp_rn(g6)));
    const float den = __fmul_rn(e4m3_to_f32(S), g);
    float q[E];
#pragma unroll
    for (int i = 0; i < E; ++i) q[i] = 0.f;
    if (S != 0u && den != 0.f) quotients(den, amax, q);
    uint32_t code[E];                                     // E2M1 code of element i
#pragma unroll
    for (int i = 0; i < E; i += 2) {
      const uint32_t byte = f32x2_to_e2m1x2(q[i], q[i + 1]);
      code[i] = byte & 0xFu;
      code[i + 1] = byte >> 4;
    }
    const int blk = lane / BL;
    if (kind == 0) {
      uint8_t* dst = chunk + static_cast<int64_t>(off) * RB + lane * (E / 2);
#pragma unroll
      for (int i = 0; i < E; i += 2) dst[i / 2] = static_cast<uint8_t>(code[i] | (code[i + 1] << 4));
      if (lane % BL == 0) chunk[static_cast<int64_t>(a.P) * D + static_cast<int64_t>(off) * SB + blk] = static_cast<uint8_t>(S);
    } else {
      // token-pair row off / 2: byte d holds element d of this token in nibble off % 2
      const int sh = 4 * (off & 1);
      uint8_t* row = chunk + static_cast<int64_t>(a.P) * RB + static_cast<int64_t>(off >> 1) * D + lane * E;
#pragma unroll
      for (int i = 0; i < E; ++i)
        row[i] = static_cast<uint8_t>((row[i] & ~(0xFu << sh)) | (code[i] << sh));
      if (lane % BL == 0)
        chunk[static_cast<int64_t>(a.P) * D + static_cast<int64_t>(a.P) * SB + static_cast<int64_t>(off >> 1) * 2 * SB +
              2 * blk + (off & 1)] = static_cast<uint8_t>(S);
    }
  } else {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float sc = div7(amax);                          // RN(amax / 7)
    uint32_t nib = 0;                                     // element i in nibble i
    if (sc != 0.f) {
      float q[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      float qe[E];
      quotients(sc, amax, qe);
#pragma unroll
      for (int i = 0; i < E; ++i) q[i] = qe[i];
      nib = int4x8(q);
    }
    if (kind == 0) {
      uint8_t* codes = chunk + static_cast<int64_t>(off) * RB + lane * (E / 2);
#pragma unroll
      for (int i = 0; i < E / 2; ++i) codes[i] = static_cast<uint8_t>(nib >> (8 * i));
    } else {
      // V: pair row off / 2, this token's 16-bit halves (elements 4k .. 4k+3
      // in the low half of word k for an even token, the high half for an
      // odd one); byte i holds elements e, e + 1 with e = lane E + 2i
      uint8_t* row = chunk + static_cast<int64_t>(a.P) * RB + static_cast<int64_t>(off >> 1) * D + 2 * (off & 1);
#pragma unroll
      for (int i = 0; i < E / 2; ++i) {
        const int e = lane * E + 2 * i;
        row[4 * (e >> 2) + ((e & 3) >> 1)] = static_cast<uint8_t>(nib >> (8 * i));
      }
    }
    if (lane == 0) reinterpret_cast<float*>(chunk + static_cast<int64_t>(a.P) * D)[static_cast<int64_t>(kind) * a.P + off] = sc;
  }
}

// The CTA's jobs, two tasks each (K, V); warp w takes tasks w, w + 4, ...
template <int D, int FMT>
__device__ __forceinline__ void run_new_token_jobs(const DecodeArgs& a, const int4* jobs, int nj) {
  for (int t = threadIdx.x >> 5; t < 2 * nj; t += kNW) write_new_token<D, FMT>(a, jobs[t >> 1], t & 1);
}

// The general form of the job list: the units whose last tile is in the
// CTA's range [c0, c1) of the global tile order, found by a scan over the
// requests in blocks of the CTA's threads, in rounds of at most one unit per
// thread (one unit index j at a time).  Ends with every job written.
template <int D, int FMT>
__device__ __forceinline__ void new_tokens_by_rounds(const DecodeArgs& a, int64_t c0, int64_t c1, int UPB,
                                                  int64_t* red, int4* jobs, int* s_njobs) {
  const int tid = threadIdx.x;
  int64_t acc = 0;
  for (int b0 = 0; b0 < a.B; b0 += kNW * 32) {
    const int b = b0 + tid;
    const int n_b = (b < a.B) ? (clamp_len(a, b, false) + kTT - 1) / kTT : 0;
    int64_t tot;
    const int64_t start = acc + block_scan(static_cast<int64_t>(n_b) * UPB, red, tot);
    acc += tot;
    const int64_t first_last = start + n_b - 1, last_last = start + static_cast<int64_t>(UPB) * n_b - 1;
    const bool some = n_b > 0 && last_last >= c0 && first_last < c1;
    if (!__syncthreads_or(some)) continue;
    for (int j = 0; j < UPB; ++j) {
      const int64_t last = start + static_cast<int64_t>(j + 1) * n_b - 1;
      const bool mine = n_b > 0 && last >= c0 && last < c1;
      if (!__syncthreads_or(mine)) continue;
      if (tid == 0) *s_njobs = 0;
      __syncthreads();
      int4 job;
      if (mine && new_token_job(a, b, j, job)) jobs[atomicAdd(s_njobs, 1)] = job;
      __syncthreads();
      run_new_token_jobs<D, FMT>(a, jobs, *s_njobs);
      __syncthreads();
    }
  }
}

// STEP: the kv4_decode_step form (the new tokens written first; NVFP4 and
// INT4 only); a separate instantiation, so the plain decode's code and
// registers are untouched.
template <int D, int FMT, bool STEP>
__global__ void __launch_bounds__(kNW * 32, kCtas)
decode4_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap cmap,
               const __grid_constant__ CUtensorMap smap) {
  using Gm = Geo4<D, FMT>;
  constexpr int RB = Gm::RB, SB = Gm::SB, KB = Gm::KB, VB = Gm::VB, MT = Gm::MT;
  grid_dep_launch();   // the combine may be scheduled now; it waits for this grid
  grid_dep_wait();     // inputs written by the previous kernel are visible
  extern __shared__ uint8_t smem_raw[];

  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int grp = lane >> 2, tig = lane & 3;
  const int ngrp = (a.G + 7) >> 3;
  const int UPB = a.Hkv * ngrp;            // units per request
  const int S = a.num_splits;

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - smem_u32(smem_raw));
  const uint32_t cring = base + Gm::OFF_C + warp * Gm::NS * Gm::STC;  // this warp's code stages
  const uint32_t sring = base + Gm::OFF_S + warp * Gm::NS * Gm::STS;  // and scale stages
  const uint32_t qsm = base + Gm::OFF_Q + lane * 16;                   // query fragment group j at + 512 j
  float* sAcc = reinterpret_cast<float*>(gbase + Gm::OFF_ACC);
  float* sMeta = reinterpret_cast<float*>(gbase + Gm::OFF_META);
  Seg* sSeg = reinterpret_cast<Seg*>(gbase + Gm::OFF_SEG);
  int64_t* sRed = reinterpret_cast<int64_t*>(gbase + Gm::OFF_RED);
  const uint32_t bars = base + Gm::OFF_BAR + warp * Gm::NS * 8;
  __shared__ int s_nseg;
  __shared__ int s_njobs;           // kv4_decode_step: new-token jobs of this CTA
  __shared__ float s_qpre;
  __shared__ long long s_cursor, s_cum, s_b;

  if (lane == 0) {
    for (int s2 = 0; s2 < Gm::NS; ++s2) mbar_init(bars + 8 * s2, 1);
    fence_mbar_init();
  }
  if (tid == 0) {
    prefetch_tensormap(&cmap);
    prefetch_tensormap(&smap);
  }
  // kv4_decode_step's jobs (at most kJobs listed here; sAcc is free until
  // the first merge).  The host allows it only with G <= 8, so unit j of a
  // request is kv head j.
  constexpr int kJobs = kNW * 32;
  static_assert(!STEP || 32 * Gm::AS * 4 >= kJobs * 16, "job list");
  int4* sJobs = reinterpret_cast<int4*>(sAcc);
  if (STEP && tid == 0) s_njobs = 0;   // before the barriers below

  // ---- this CTA's tile range [cursor, c1) in the global (b, unit, tile) order ------
  int64_t T = 0, c1 = 0;
  if (a.unit_ctas) {
    const int u = blockIdx.x, b = u / UPB;
    const int n_u = (clamp_len(a, b, tid == 0) + kTT - 1) / kTT;
    if (tid == 0) {
      sSeg[0] = Seg{u, 0, n_u, 0, clamp_len(a, b, false)};
      s_nseg = 1;
      int4 job;
      if (STEP && new_token_job(a, b, u - b * UPB, job)) {
        sJobs[0] = job;
        s_njobs = 1;
      }
    }
  } else {
    int64_t ex0 = 0, v0 = 0;          // this thread's request when B <= kJobs
    for (int b0 = 0; b0 < a.B; b0 += kNW * 32) {
      const int b = b0 + tid;
      const int64_t v = (b < a.B) ? static_cast<int64_t>((clamp_len(a, b, blockIdx.x == 0) + kTT - 1) / kTT) * UPB : 0;
      int64_t tot;
      const int64_t ex = block_scan(v, sRed, tot);
      if (blockIdx.x == 0 && b < a.B) a.cum[b] = T + ex;        // for combine_kernel
      if (b0 == 0) {
        ex0 = ex;
        v0 = v;
      }
      T += tot;
    }
    if (blockIdx.x == 0 && tid == 0) a.cum[a.B] = T;
    c1 = part_begin4(blockIdx.x + 1, T, a.n_cta);
    const int64_t c0 = part_begin4(blockIdx.x, T, a.n_cta);
    if (tid == 0) s_cursor = c0;
    if constexpr (STEP) {
      // the units of this thread's request whose last tile is in [c0, c1)
      if (a.B <= kJobs && v0 > 0) {
        const int64_t n_b = v0 / UPB;
        bool have = false;
        int4 job;
        for (int j = 0; j < UPB; ++j) {
          const int64_t last = ex0 + (j + 1) * n_b - 1;
          if (last < c0 || last >= c1) continue;
          if (!have && !new_token_job(a, tid, 0, job)) break;
          have = true;
          job.y = j;
          const int k = atomicAdd(&s_njobs, 1);
          if (k < kJobs) sJobs[k] = job;
        }
      }
    }
  }
  __syncthreads();
  if constexpr (STEP) {
    const int nj = s_njobs;
    if ((!a.unit_ctas && a.B > kJobs) || nj > kJobs) {
      __syncthreads();                // every thread has read s_njobs
      new_tokens_by_rounds<D, FMT>(a, part_begin4(blockIdx.x, T, a.n_cta), c1, UPB, sRed, sJobs, &s_njobs);
      asm volatile("fence.proxy.async.global;" ::: "memory");
      __syncthreads();
    } else if (nj > 0) {
      run_new_token_jobs<D, FMT>(a, sJobs, nj);
      // the generic-proxy writes of the pool before this CTA's TMA reads of it
      asm volatile("fence.proxy.async.global;" ::: "memory");
      __syncthreads();
    }
  }

  // ---- per-thread shared-memory offsets inside a stage ----------------------
  // K: bytes [KB tig, KB (tig + 1)) of token rows grp and grp + 8, in 16-byte
  // units with their own swizzled offsets (a TMA swizzle pattern repeats every
  // 8 rows, so row grp + 8 is the same offset plus 8 rows).
  const uint32_t k_off0 = swz<RB>(grp, KB * tig);
  const uint32_t k_off1 = swz<RB>(grp, KB * tig + 16);
  const uint32_t ks_off = grp * SB + (D / 64) * tig;                 // K scale bytes of row grp
  // NVFP4 V (token-pair rows: byte d of pair row p holds dim d of tokens 2p,
  // 2p+1): head dims [D0, D0 + D/8) of pairs tig and tig + 4; the dim chunks
  // go to groups in the order 4 (grp & 1) + grp/2 so the two groups of a
  // quarter-warp read pair-row halves of opposite parity (distinct banks).
  constexpr int D0S = D / 8;
  const int D0 = D0S * (4 * (grp & 1) + (grp >> 1));
  const uint32_t vp_off0 = Gm::CSK + swz<RB>(2 * tig + D0 / RB, D0 % RB);
  const uint32_t vp_off1 = Gm::CSK + swz<RB>(2 * tig + D0 / RB, D0 % RB + 16);
  const uint32_t vps_off = kTT * SB + tig * (D / 8) + 2 * (D0 / 16);
  // INT4 and k8v4 V take the same pair-row offsets (word j of a pair row
  // holds dims 4j .. 4j+3 of both tokens); V starts after the tile's K
  // bytes (CSK = CS but for k8v4, whose FP8 key rows are D bytes).
  // k8v4 K (FP8, KH lines of KHB bytes a token): the 16-byte units of bytes
  // [KB tig, KB (tig + 1)) of token grp; token grp + 8 is 8 KRB bytes on (the
  // swizzle pattern repeats every 8 lines).
  constexpr int KU = Gm::K8 ? Gm::KB / 16 : 1;
  uint32_t k8_off[KU];
#pragma unroll
  for (int u = 0; u < KU; ++u) {
    const int byte = Gm::KB * tig + 16 * u;
    k8_off[u] = swz<Gm::KHB>(grp * Gm::KH + byte / Gm::KHB, byte % Gm::KHB);
  }

  const uint64_t pol = policy_evict_first();
  int issued = 0, consumed = 0;     // warp-local tile counters
  int islot = 0, cslot = 0;         // ring slots of the next tile to issue / consume
  uint32_t cphase = 0;              // phase parity of the consume slot's barrier
  bool timed_out = false;

  // passes over the CTA range, kMaxSeg segments at a time
  while (true) {
    if (!a.unit_ctas) {
      const int64_t cur = s_cursor;
      __syncthreads();
      if (cur >= c1) break;
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
          const int split = static_cast<int>(part_of4(t, n_u, S));
          const int64_t send = part_begin4(split + 1, n_u, S);
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

    // this warp's run of tiles inside segment k
    auto my_run = [&](int k, int& beg, int& cnt) {
      const int n = sSeg[k].n;
      const int q = (n + kNW - 1) / kNW;
      beg = min(n, warp * q);
      cnt = min(n, beg + q) - beg;
    };

    // ---- issue cursor over this pass's segments, with its block-table cache ----
    int ks = -1, io = 0, is_bg = 0, is_cn = 0, is_t0 = 0, is_h = 0;
    int i_pass = 0, i_total = 0;
    for (int k = 0; k < nseg; ++k) {
      int bg, cn;
      my_run(k, bg, cn);
      i_total += cn;
    }
    int p_first = 0, p_last = -1, win = 0, pg_cur = 0, pg_nxt = 0;
    int pi = 0, po = 0;               // page index and offset of the next tile's first token
    int c_pi = -1;                    // page whose TMA bases are cached below
    uint32_t c_row = 0;               // code-row index of that page-head chunk (k8v4: the chunk index)
    uint32_t c_srow = 0;              // scale-row index (16 SB bytes a row) of its K scales
    const uint8_t* c_vs = nullptr;    // k8v4: the chunk's V scales
    const int32_t* bt = a.block_table;

    auto issue = [&]() {      // warp-uniform; issues the next tile of this pass
      while (io >= is_cn) {   // enter the next segment with tiles for this warp
        ++ks;
        io = 0;
        my_run(ks, is_bg, is_cn);
        const Seg sg = sSeg[ks];
        const int b = sg.u / UPB;
        is_h = (sg.u % UPB) / ngrp;
        is_t0 = sg.t0;
        if (is_cn > 0) {        // reload the page cache for this run
          const int tf = (sg.t0 + is_bg) * kTT;
          pi = tf / a.P;
          po = tf - pi * a.P;
          p_first = pi;
          p_last = (min(sg.len, (sg.t0 + is_bg + is_cn) * kTT) - 1) / a.P;
          win = 0;
          c_pi = -1;
          bt = a.block_table + static_cast<int64_t>(b) * a.max_pages;
          const int r0 = p_first + lane, r1 = p_first + 32 + lane;
          pg_cur = r0 <= p_last ? __ldg(bt + r0) : 0;
          pg_nxt = r1 <= p_last ? __ldg(bt + r1) : 0;
        }
      }
      if (pi != c_pi) {       // a new page: its chunk's TMA row and scale address
        while (((pi - p_first) >> 5) > win) {
          ++win;
          pg_cur = pg_nxt;
          const int r = p_first + (win + 1) * 32 + lane;
          pg_nxt = r <= p_last ? __ldg(bt + r) : 0;
        }
        const int rel = pi - p_first;
        const int pc = __shfl_sync(kFull, pg_cur, rel & 31), pn = __shfl_sync(kFull, pg_nxt, rel & 31);
        int page = ((rel >> 5) == win) ? pc : pn;
        if (page < 0 || page >= a.num_pages) {
          if (lane == 0) set_error(a.err, KV4_EBOUNDS);
          page = 0;
        }
        const int64_t ci = static_cast<int64_t>(page) * a.Hkv + is_h;
        const int64_t chunk = ci * a.chunk_bytes;
        if constexpr (Gm::K8) {
          c_row = static_cast<uint32_t>(ci);
          c_vs = a.pool + chunk + static_cast<int64_t>(a.P) * (Gm::KRB + RB);
        } else {
          c_row = static_cast<uint32_t>(chunk / RB);
          c_srow = static_cast<uint32_t>((chunk + static_cast<int64_t>(a.P) * 2 * RB) / (kTT * SB));
        }
        c_pi = pi;
      }
      if (lane == 0) {
        const uint32_t cst = cring + islot * Gm::STC, sst = sring + islot * Gm::STS;
        const uint32_t bar = bars + 8 * islot;
        mbar_arrive_expect_tx(bar, Gm::STC + Gm::STS);
        if constexpr (Gm::K8) {
          // the tile's K lines (4-D box: line, half, token, chunk), its V rows
          // (3-D: row, token, chunk) and its 16 V scales (a 64-byte bulk copy)
          tma_load_4d(cst, &cmap, 0, 0, po, static_cast<int>(c_row), bar, pol);
          tma_load_3d(cst + Gm::CSK, &smap, 0, po, static_cast<int>(c_row), bar, pol);
          bulk_load(sst, c_vs + 4 * po, Gm::STS, bar, pol);
        } else {
          // the tile's K and V code rows (one 3-D box), then its K and V scale rows
          tma_load_3d(cst, &cmap, 0, static_cast<int>(c_row) + po, 0, bar, pol);
          tma_load_3d(sst, &smap, 0, static_cast<int>(c_srow) + po / kTT, 0, bar, pol);
        }
      }
      islot = (islot + 1 == Gm::NS) ? 0 : islot + 1;
      po += kTT;                       // a tile never straddles a page: 16 divides P
      if (po == a.P) { po = 0; ++pi; }
      ++io;
      ++issued;
      ++i_pass;
    };

    for (int k0 = 0; k0 < Gm::NS && i_pass < i_total && !timed_out; ++k0) issue();

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

      // ---- the unit's query fragments (B operand of S^T = K q^T), once per CTA ----
      // Thread (grp, tig) of any warp uses query row g0 + grp, dims
      // [2 KB tig, 2 KB (tig + 1)); warp 0 converts them (bf16 -> f16, |q|
      // pre-scaled by an exact power of two into f16 range) into shared memory.
      if constexpr (Gm::K8) {
        // q_rot = S_D q (the Walsh-Hadamard butterflies in FP32; the 1/sqrt(D)
        // goes into qk_scale), built for the unit's heads in the merge buffer
        float* qs = sAcc;
        for (int e = tid; e < 8 * D; e += kNW * 32) {
          const int g = e / D;
          qs[e] = (g < ng) ? __bfloat162float(a.q[(static_cast<int64_t>(b) * a.Hq + hq0 + g) * D + e % D]) : 0.f;
        }
        for (int len = 1; len < D; len <<= 1) {
          __syncthreads();
          for (int p2 = tid; p2 < 8 * (D / 2); p2 += kNW * 32) {
            const int vec = p2 / (D / 2), r = p2 % (D / 2);
            float* v = qs + vec * D + (r / len) * 2 * len + (r % len);
            const float x0 = v[0], x1 = v[len];
            v[0] = __fadd_rn(x0, x1);
            v[len] = __fsub_rn(x0, x1);
          }
        }
        __syncthreads();
        // |q_rot| pre-scaled into f16 range by an exact power of two
        float qmax = 0.f;
        for (int e = tid; e < 8 * D; e += kNW * 32) qmax = fmaxf(qmax, fabsf(qs[e]));
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) qmax = fmaxf(qmax, __shfl_xor_sync(kFull, qmax, o2));
        if (lane == 0) sMeta[warp] = qmax;
        __syncthreads();
        qmax = fmaxf(fmaxf(sMeta[0], sMeta[1]), fmaxf(sMeta[2], sMeta[3]));
        float qpre = 1.f;
        if (qmax > 16384.f) {
          int e;
          frexpf(qmax / 16384.f, &e);
          qpre = ldexpf(1.f, -e);
        }
        // B fragments of k-step j: head grp, dims KB tig + 4j .. + 3 (the dims
        // of the lane's K word j), q_rot as f16 hi + lo
        for (int j = warp; j < Gm::KS; j += kNW) {
          const float* qq = qs + grp * D + KB * tig + 4 * j;
          uint32_t hi[2], lo[2];
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            const float v0 = qq[2 * e2] * qpre, v1 = qq[2 * e2 + 1] * qpre;
            hi[e2] = pack_f16x2(v0, v1);
            const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hi[e2]));
            lo[e2] = pack_f16x2(v0 - hf.x, v1 - hf.y);
          }
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};"
                       :: "r"(qsm + j * 512), "r"(hi[0]), "r"(hi[1]), "r"(lo[0]), "r"(lo[1]) : "memory");
        }
        if (tid == 0) s_qpre = qpre;
      } else if (warp == 0) {
        constexpr int NG = KB / 4;
        uint4 raw[NG];
        const bool row_ok = grp < ng;
        const __nv_bfloat16* qrow = a.q + (static_cast<int64_t>(b) * a.Hq + hq0 + grp) * D + 2 * KB * tig;
#pragma unroll
        for (int i = 0; i < NG; ++i)
          raw[i] = row_ok ? __ldg(reinterpret_cast<const uint4*>(qrow + 8 * i)) : make_uint4(0, 0, 0, 0);
        float qmax = 0.f;
#pragma unroll
        for (int i = 0; i < NG; ++i) {
          const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&raw[i]);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 f = __bfloat1622float2(p2[j]);
            qmax = fmaxf(qmax, fmaxf(fabsf(f.x), fabsf(f.y)));
          }
        }
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) qmax = fmaxf(qmax, __shfl_xor_sync(kFull, qmax, o2));
        float qpre = 1.f;
        if (qmax > 16384.f) {
          int e;
          frexpf(qmax / 16384.f, &e);
          qpre = ldexpf(1.f, -e);
        }
#pragma unroll
        for (int i = 0; i < NG; ++i) {
          float e[8];
          const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&raw[i]);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 f = __bfloat1622float2(p2[j]);
            e[2 * j] = f.x * qpre;
            e[2 * j + 1] = f.y * qpre;
          }
          uint32_t w0, w1, w2, w3;
          if constexpr (FMT == KV4_NVFP4) {
            // k-step: k (2tig, 2tig+1) <-> dims {0,1} of a 4-dim group, (2tig+8, +9) <-> {2,3}
            w0 = pack_f16x2(e[0], e[1]); w1 = pack_f16x2(e[2], e[3]);
            w2 = pack_f16x2(e[4], e[5]); w3 = pack_f16x2(e[6], e[7]);
          } else {
            // INT4 nibble order: (e0,e4), (e1,e5) for one k-step; (e2,e6), (e3,e7) for the next
            w0 = pack_f16x2(e[0], e[4]); w1 = pack_f16x2(e[1], e[5]);
            w2 = pack_f16x2(e[2], e[6]); w3 = pack_f16x2(e[3], e[7]);
          }
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};"
                       :: "r"(qsm + i * 512), "r"(w0), "r"(w1), "r"(w2), "r"(w3) : "memory");
        }
        if (lane == 0) s_qpre = qpre;
      }
      __syncthreads();
      // NVFP4: g_K; k8v4: s_K and the rotation's 1/sqrt(D); INT4: per token below
      const float qk_scale = a.sm_scale * ((FMT != KV4_INT4_PTH) ? __ldg(a.gscale) : 1.f) *
                             (Gm::K8 ? rsqrtf(static_cast<float>(D)) : 1.f) * 1.4426950408889634f / s_qpre;

      // ---- running softmax state, heads g0 + 2tig + c, c = 0, 1 -------------------
      float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
      float sref = 0.f;       // INT4: largest V scale seen
      float inv_sref = 1.f;   // and 1 / s_ref (1 until s_ref > 0)
      float o[MT][4];
#pragma unroll
      for (int mi = 0; mi < MT; ++mi) o[mi][0] = o[mi][1] = o[mi][2] = o[mi][3] = 0.f;

      for (int jt = 0; jt < cn && !timed_out; ++jt) {
        const uint32_t st = cring + cslot * Gm::STC, sst = sring + cslot * Gm::STS;
        if (!mbar_wait_bounded(bars + 8 * cslot, cphase)) {
          // give the copies still in flight a bounded chance to land, then stop
          for (int j = consumed + 1; j < issued; ++j) mbar_wait_bounded(bars + 8 * (j % Gm::NS), (j / Gm::NS) & 1);
          timed_out = true;
          break;
        }
        const int t0 = (sg.t0 + bg + jt) * kTT;
        const int valid = min(kTT, L - t0);

        // -------- S^T[t][g] = K q^T: 16 tokens x 8 heads, two accumulation chains --------
        // sacc: c0 = (token grp, head 2tig), c1 = (grp, 2tig+1), c2 = (grp+8, 2tig), c3 = (grp+8, 2tig+1)
        float sacc[2][4];
        sacc[0][0] = sacc[0][1] = sacc[0][2] = sacc[0][3] = 0.f;
        sacc[1][0] = sacc[1][1] = sacc[1][2] = sacc[1][3] = 0.f;
        {
          if constexpr (Gm::K8) {
            // FP8 keys are exact in f16: one word (4 dims) of each row per
            // k-step, against q_rot hi (chain 0) and lo (chain 1)
#pragma unroll
            for (int u = 0; u < KU; ++u) {
              const uint4 x0 = lds128(st + k8_off[u]), x1 = lds128(st + k8_off[u] + 8 * Gm::KRB);
              const uint32_t w0[4] = {x0.x, x0.y, x0.z, x0.w}, w1[4] = {x1.x, x1.y, x1.z, x1.w};
#pragma unroll
              for (int jj = 0; jj < 4; ++jj) {
                uint32_t a0, a1, a2, a3;
                e4m3x4_to_f16x2x2(w0[jj], a0, a2);
                e4m3x4_to_f16x2x2(w1[jj], a1, a3);
                const uint4 qv = lds128(qsm + (4 * u + jj) * 512);
                mma_f16_16816(sacc[0], a0, a1, a2, a3, qv.x, qv.y);
                mma_f16_16816(sacc[1], a0, a1, a2, a3, qv.z, qv.w);
              }
            }
          }
          // KCW code words of each row at a time (word c of the thread's KB bytes
          // sits at byte 4 (c % 4) of 16-byte unit c / 4)
          constexpr int W = Gm::K8 ? 0 : KB / 4, CW = KCW < W ? KCW : (W > 0 ? W : 1);
          uint32_t hs[2][4];         // NVFP4: f16x2 broadcasts of the row's blocks
          if constexpr (FMT == KV4_NVFP4) {
#pragma unroll
            for (int r = 0; r < 2; ++r) {
              const uint32_t sraw = load_scale_bytes<D / 64>(sst + ks_off + 8 * SB * r);
              e4m3x4_to_f16x2x2(prmt(sraw, 0u, 0x1100u), hs[r][0], hs[r][1]);
              if constexpr (D / 64 > 2) e4m3x4_to_f16x2x2(prmt(sraw, 0u, 0x3322u), hs[r][2], hs[r][3]);
            }
          }
#pragma unroll
          for (int c0 = 0; c0 < W; c0 += CW) {
            uint32_t kw0[CW], kw1[CW];
            const uint32_t ko = st + ((c0 >> 2) ? k_off1 : k_off0) + 4 * (c0 & 3);
            load_bytes<4 * CW>(ko, kw0);
            load_bytes<4 * CW>(ko + 8 * RB, kw1);
#pragma unroll
            for (int jj = 0; jj < CW; ++jj) {
              const uint4 qv = lds128(qsm + (c0 + jj) * 512);
              if constexpr (FMT == KV4_NVFP4) {
                uint32_t e0[4], e1[4];
                e2m1x8_to_f16x2x4(kw0[jj], e0);
                e2m1x8_to_f16x2x4(kw1[jj], e1);
                const uint32_t s0 = hs[0][(c0 + jj) >> 1], s1 = hs[1][(c0 + jj) >> 1];
                mma_f16_16816(sacc[0], hmul2(e0[0], s0), hmul2(e1[0], s1), hmul2(e0[1], s0), hmul2(e1[1], s1),
                              qv.x, qv.y);
                mma_f16_16816(sacc[1], hmul2(e0[2], s0), hmul2(e1[2], s1), hmul2(e0[3], s0), hmul2(e1[3], s1),
                              qv.z, qv.w);
              } else {
                const uint32_t w0 = kw0[jj], w1 = kw1[jj];
                mma_f16_16816(sacc[0], int4_lo_pair(w0), int4_lo_pair(w1), int4_hi_pair(w0), int4_hi_pair(w1),
                              qv.x, qv.y);
                const uint32_t y0 = w0 >> 8, y1 = w1 >> 8;
                mma_f16_16816(sacc[1], int4_lo_pair(y0), int4_lo_pair(y1), int4_hi_pair(y0), int4_hi_pair(y1),
                              qv.z, qv.w);
              }
            }
          }
        }
        // x[2r + c]: token grp + 8r, head 2tig + c (base-2 logits)
        float x[4];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          float sk = 1.f;
          if constexpr (FMT == KV4_INT4_PTH) sk = __uint_as_float(lds32(sst + 4 * (grp + 8 * r)));
#pragma unroll
          for (int c = 0; c < 2; ++c) x[2 * r + c] = (sacc[0][2 * r + c] + sacc[1][2 * r + c]) * (qk_scale * sk);
        }
        if (valid < kTT) {
          // tokens past the end get no weight (their rows may hold anything)
#pragma unroll
          for (int r = 0; r < 2; ++r)
            if (grp + 8 * r >= valid) x[2 * r] = x[2 * r + 1] = -INFINITY;
        }

        // -------- online softmax with a lazily raised base --------
        // One vote a tile: only when a logit tops its head's base by more than
        // kLazy (or, INT4, a V scale tops s_ref) are the bases raised and O,
        // l rescaled.
        float sv[2];
        float smax = 0.f;
        if constexpr (Gm::PTV) {
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int t = grp + 8 * r;
            const float v = __uint_as_float(lds32(sst + Gm::VS + 4 * t));
            sv[r] = (t < valid && v > 0.f) ? v : 0.f;     // NaN, <= 0 and past the end: no weight
            smax = fmaxf(smax, sv[r]);
          }
        }
        float tmx[2] = {fmaxf(x[0], x[2]), fmaxf(x[1], x[3])};
        bool raise = tmx[0] > m_run[0] + kLazy || tmx[1] > m_run[1] + kLazy;
        if constexpr (Gm::PTV) raise = raise || smax > sref;
        if (__any_sync(kFull, raise)) {
          float corr_o[2] = {1.f, 1.f};
          if constexpr (Gm::PTV) {
#pragma unroll
            for (int o2 = 4; o2 < 32; o2 <<= 1) smax = fmaxf(smax, __shfl_xor_sync(kFull, smax, o2));
            if (smax > sref) {
              corr_o[0] = corr_o[1] = (sref > 0.f) ? sref / smax : 0.f;
              sref = smax;
              inv_sref = 1.f / sref;
            }
          }
#pragma unroll
          for (int c = 0; c < 2; ++c) {
#pragma unroll
            for (int o2 = 4; o2 < 32; o2 <<= 1) tmx[c] = fmaxf(tmx[c], __shfl_xor_sync(kFull, tmx[c], o2));
            const float mnew = fmaxf(m_run[c], tmx[c]);
            if (mnew > m_run[c]) {
              const float cr = fast_exp2(m_run[c] - mnew);     // 0 when m_run == -inf
              l_run[c] *= cr;
              corr_o[c] *= cr;
              m_run[c] = mnew;
            }
          }
#pragma unroll
          for (int mi = 0; mi < MT; ++mi) {
            o[mi][0] *= corr_o[0]; o[mi][1] *= corr_o[1]; o[mi][2] *= corr_o[0]; o[mi][3] *= corr_o[1];
          }
        }
        // weights and their f16 hi + lo split, transposed into the P^T B operand:
        // b0 <- tokens (2tig, 2tig+1) of head grp, b1 <- tokens (8+2tig, 8+2tig+1)
        uint32_t pb[2], pl[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          float w[2];
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            // m_run is finite here: every tile has a valid first token, and the
            // run's first tile raised it from -inf
            const float p = fast_exp2(x[2 * r + c] - m_run[c]);
            l_run[c] += p;
            w[c] = p;
            if constexpr (Gm::PTV) w[c] = p * (sv[r] * inv_sref);
          }
          const uint32_t hi = pack_f16x2(w[0], w[1]);
          const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hi));
          const uint32_t lo = pack_f16x2(w[0] - hf.x, w[1] - hf.y);
          pb[r] = movmatrix_trans(hi);
          pl[r] = movmatrix_trans(lo);
        }

        // -------- O^T += V^T P^T --------
        const int ta = 2 * tig;                   // tokens ta, ta+1 (k 2tig..) and ta+8, ta+9
        if constexpr (FMT == KV4_NVFP4) {
          constexpr int NSB = (D0S >= 32) ? 4 : 2;
          const uint32_t xab = load_scale_bytes<NSB>(sst + vps_off);
          const uint32_t xcd = load_scale_bytes<NSB>(sst + vps_off + D / 2);
          uint32_t sab[2], scd[2];
          e4m3x4_to_f16x2x2(xab, sab[0], sab[1]);
          e4m3x4_to_f16x2x2(xcd, scd[0], scd[1]);
          if (valid < kTT) {
            // a zero scale zeroes the (finite) codes of tokens past the end
            const uint32_t mab = ((ta < valid) ? 0xFFFFu : 0u) | ((ta + 1 < valid) ? 0xFFFF0000u : 0u);
            const uint32_t mcd = ((ta + 8 < valid) ? 0xFFFFu : 0u) | ((ta + 9 < valid) ? 0xFFFF0000u : 0u);
            sab[0] &= mab; sab[1] &= mab;
            scd[0] &= mcd; scd[1] &= mcd;
          }
          constexpr int W = D0S / 4, CW = VCW < W ? VCW : W;
#pragma unroll
          for (int c0 = 0; c0 < W; c0 += CW) {
            const uint32_t vo = st + ((c0 >> 2) ? vp_off1 : vp_off0) + 4 * (c0 & 3);
            uint32_t wab[CW], wcd[CW];
            load_bytes<4 * CW>(vo, wab);
            load_bytes<4 * CW>(vo + 8 * RB, wcd);
#pragma unroll
            for (int jj = 0; jj < CW; ++jj) {
              const int j = c0 + jj;
              uint32_t f[4], hh4[4];
              e2m1x8_to_f16x2x4(wab[jj], f);
              e2m1x8_to_f16x2x4(wcd[jj], hh4);
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                const int mi = 2 * j + hh;                 // dims D0 + 2mi, D0 + 2mi + 1
                const int bj = (VB >= 8) ? mi / 8 : 0;     // block of this m-tile among the thread's
                const uint32_t a0 = hmul2(f[2 * hh], sab[bj]);
                const uint32_t a1 = hmul2(f[2 * hh + 1], sab[bj]);
                const uint32_t a2 = hmul2(hh4[2 * hh], scd[bj]);
                const uint32_t a3 = hmul2(hh4[2 * hh + 1], scd[bj]);
                mma_f16_16816(o[mi], a0, a1, a2, a3, pb[0], pb[1]);
                mma_f16_16816(o[mi], a0, a1, a2, a3, pl[0], pl[1]);
              }
            }
          }
        } else {
          // INT4 / k8v4 V in token-pair rows, by 16-bit halves: word j of
          // the thread's span holds dims D0 + 4j .. 4j+3 of both tokens, so a
          // shift by 0 or 8 bits lines up two dims of the two tokens in the
          // halves; the per-token V scale rides on the weight
          constexpr int W = D0S / 4, CW = VCW < W ? VCW : W;
#pragma unroll
          for (int c0 = 0; c0 < W; c0 += CW) {
            const uint32_t vo = st + ((c0 >> 2) ? vp_off1 : vp_off0) + 4 * (c0 & 3);
            uint32_t wab[CW], wcd[CW];
            load_bytes<4 * CW>(vo, wab);
            load_bytes<4 * CW>(vo + 8 * RB, wcd);
#pragma unroll
            for (int jj = 0; jj < CW; ++jj) {
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                const int mi = 2 * (c0 + jj) + hh;         // dims D0 + 2mi, D0 + 2mi + 1
                const uint32_t xa = hh ? wab[jj] >> 8 : wab[jj];
                const uint32_t xc = hh ? wcd[jj] >> 8 : wcd[jj];
                const uint32_t a0 = int4_lo_pair(xa), a1 = int4_hi_pair(xa);
                const uint32_t a2 = int4_lo_pair(xc), a3 = int4_hi_pair(xc);
                mma_f16_16816(o[mi], a0, a1, a2, a3, pb[0], pb[1]);
                mma_f16_16816(o[mi], a0, a1, a2, a3, pl[0], pl[1]);
              }
            }
          }
        }
        __syncwarp();
        ++consumed;
        cslot = (cslot + 1 == Gm::NS) ? 0 : cslot + 1;
        if (cslot == 0) cphase ^= 1u;
        if (i_pass < i_total) issue();     // refill the stage just freed
      }
      // A warp that timed out stops streaming but still joins every merge below,
      // so the CTA's barriers stay matched; its partial state is empty.
      if (timed_out) {
        m_run[0] = m_run[1] = -INFINITY;
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
          const bool some = l_run[c] > 0.f;
          float my = m_run[c];
          if constexpr (Gm::PTV) my = (sref > 0.f) ? m_run[c] + fast_log2(sref) : -INFINITY;
          mt[0] = some ? m_run[c] : -INFINITY;
          mt[1] = some ? my : -INFINITY;
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
      // k8v4 rotates the merged output back in the combine: always pieces
      const bool direct = !Gm::K8 && (a.unit_ctas || (S == 1 && sg.t0 == 0 && sg.n == (L + kTT - 1) / kTT));
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
        // (d, g) lives in lane (grp, tig) with tig = g/2 and grp the group that
        // holds dim chunk q = (d/2) / VB (pi^-1(q) for every format), in
        // o[mi][g%2] with mi = (d/2) % VB; d+1 in o[mi][g%2 + 2]; d+2, d+3 in o[mi+1].
        const int hd = d >> 1, mi = hd % VB, c = g & 1;
        const int q = hd / VB, gq = 2 * (q & 3) + (q >> 2);
        const float* row = sAcc + (gq * 4 + (g >> 1)) * Gm::AS + 4 * mi + c;
        const float4 acc = make_float4(row[0], row[2], row[4], row[6]);
        if (direct) {
          const float gv = (FMT == KV4_NVFP4) ? __ldg(a.gscale + 1) : 1.f;
          const float inv = (l > 0.f && My != -INFINITY) ? gv * fast_exp2(My - Mx) / l : 0.f;
          const int64_t orow = static_cast<int64_t>(b) * a.Hq + hq0 + g;
          store_out4(a.out, a.out_f32, orow * D + d, make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
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

// ------------------------------------------------------------------ launch
template <int D, int FMT, bool STEP = false>
static cudaError_t launch4(const DecodeArgs& a, const CUtensorMap& cmap, const CUtensorMap& smap,
                           cudaStream_t st) {
  using Gm = Geo4<D, FMT>;
  auto* k = decode4_kernel<D, FMT, STEP>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Gm::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_cta);
  cfg.blockDim = dim3(kNW * 32);
  cfg.dynamicSmemBytes = Gm::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, a, cmap, smap);
}

int decode4_ctas_per_sm() { return kCtas; }

cudaError_t launch_decode4(const DecodeArgs& a, const CUtensorMap& cmap, const CUtensorMap& smap,
                           cudaStream_t st) {
  if (a.fmt == KV4_K8V4) {
    switch (a.D) {
      case 64: return launch4<64, KV4_K8V4>(a, cmap, smap, st);
      case 128: return launch4<128, KV4_K8V4>(a, cmap, smap, st);
      default: return launch4<256, KV4_K8V4>(a, cmap, smap, st);
    }
  }
  const bool step = a.k_new != nullptr;
  if (a.fmt == KV4_NVFP4) {
    switch (a.D) {
      case 64: return step ? launch4<64, KV4_NVFP4, true>(a, cmap, smap, st) : launch4<64, KV4_NVFP4>(a, cmap, smap, st);
      case 128:
        return step ? launch4<128, KV4_NVFP4, true>(a, cmap, smap, st) : launch4<128, KV4_NVFP4>(a, cmap, smap, st);
      default:
        return step ? launch4<256, KV4_NVFP4, true>(a, cmap, smap, st) : launch4<256, KV4_NVFP4>(a, cmap, smap, st);
    }
  }
  switch (a.D) {
    case 64:
      return step ? launch4<64, KV4_INT4_PTH, true>(a, cmap, smap, st) : launch4<64, KV4_INT4_PTH>(a, cmap, smap, st);
    case 128:
      return step ? launch4<128, KV4_INT4_PTH, true>(a, cmap, smap, st) : launch4<128, KV4_INT4_PTH>(a, cmap, smap, st);
    default:
      return step ? launch4<256, KV4_INT4_PTH, true>(a, cmap, smap, st) : launch4<256, KV4_INT4_PTH>(a, cmap, smap, st);
  }
}

}  // namespace kv4
