// Chunked-prefill / extend attention over the FP8 workspace plus the FP8
// current chunk ("SGLang's 4-bit KV cache", Figure 2, right-hand column: the
// cached prefix has been turned into FP8 in a reused buffer, and the chunk's
// queries attend over that prefix and the chunk itself).  Chunk query i of a
// request sits at position Lp + i and sees all Lp prefix keys and the chunk
// keys 0..i.  One per-tensor FP8 scale pair {s_K, s_V} serves both.
//
// This is the dense part of the path, so it runs on the fifth-generation
// tensor cores: tcgen05.mma kind::f16, accumulators in tensor memory (TMEM).
// One CTA owns 128 query rows of one query head (the MMA's M) and streams the
// request's keys in tiles of 64:
//
//   warps 0-3   softmax, one thread per query row (= TMEM lane): Q into TMEM
//               at the start; per tile S from TMEM, mask, online softmax in
//               the log2 domain, P (f16 hi + lo) back into TMEM over its own S, the
//               rare rescale of O in TMEM; the epilogue.
//   warps 4-11  converters: FP8 K and V rows from global memory (two
//               register sets, one tile of loads in flight) to f16 tiles in the 128-byte-swizzled layout the MMA reads,
//               three shared-memory stages each for K and V, freed by the
//               MMA reading them.
//   warp 13     one lane keeps an L2 bulk prefetch of the K / V rows a few
//               tiles ahead of the converters.
//   warp 12     TMEM allocation and, on one lane, the MMA issue:
//               S_j = Q K_j^T (M128 N64, K = head_dim; A = Q in TMEM) and
//               O += P_j V_j (M128 N=head_dim K64, hi then lo; A = P in TMEM), each issued
//               as soon as its operands are ready.
//
// Keeping Q and P in TMEM leaves the shared-memory data path to the K / V
// tiles (the converters' stores and the MMAs' B reads), which is what bounds
// this kernel once the tensor pipe is fed.
//
// Operand layouts.  Shared memory, K-major rows of 128 bytes in 8-row swizzle
// atoms of 1024 bytes (16-byte unit index XOR row % 8):
//   K  f16 [D/64][64 keys][64]   B of S (K-major; 8-key groups 1024 bytes apart)
//   V  f16 [D/64][64 keys][64]   B of O, MN-major: N = head_dim runs along the
//                                rows; 64-column blocks are the leading-byte-
//                                offset stride (64*128), 8-key groups the
//                                stride-byte-offset (1024)
// TMEM (lane = query row; 32-bit columns):
//   S_j  FP32, 64 columns at (j % 2) * 64;  P_j as f16 pairs over them: the
//        hi part in the first 32 columns, the lo part (p - hi) in the last 32
//   Q    f16 pairs (elements 2c, 2c+1 in column c), D/2 columns at 128
//   O    FP32, D columns at 256 (192 for head_dim 64)
// S_{j+2} reuses the columns of P_j; it is issued after O += P_j V_j, and
// tcgen05.mma operations of one thread execute in issue order.
//
// FP8 -> f16 with the hardware conversion (exact: every E4M3 value is an f16
// value).  Q is converted bf16 -> f16 once per CTA (exact for
// 2^-14 <= |q| <= 65504; larger magnitudes are flagged).  P goes to the PV
// product as an f16 hi + lo pair (the two roundings leave about 2^-22 of p);
// S and O accumulate in FP32.
//
// The maximum used for exponentiation is raised only when a tile's maximum
// exceeds it by more than 8 (log2 units), so P stays below 2^8 and O is
// rescaled in TMEM rarely; the final division by the row sum uses the same
// maximum, so the result does not depend on when the rescales happened.
// Every wait is bounded: on expiry the kernel records KV4_ETIMEOUT and winds
// down without leaving an MMA in flight past the TMEM release.
#include <cstdint>

#include "kv4_device.cuh"
#include "kv4_internal.h"

namespace kv4 {
namespace {

constexpr int kQT = 128;          // query rows per CTA (MMA M)
constexpr int kKT = 64;           // keys per tile
constexpr int kNST = 3;           // shared-memory stages for K and for V
constexpr int kThreads = 448;     // 4 softmax, 8 converter, 1 MMA and 1 prefetch warp
constexpr int kConv = 256;        // converter threads
constexpr int kMmaWarp = 12;
constexpr int kPrefetchWarp = 13;
constexpr int kPrefetchAhead = 6;  // tiles the L2 prefetch runs ahead of the converters
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct ExtGeo {
  static constexpr int KV_BYTES = kKT * D * 2;
  static constexpr int OFF_V = kNST * KV_BYTES;
  static constexpr int SMEM = 2 * kNST * KV_BYTES + 1024;     // + alignment slack
  static constexpr int S_COL = 0;                             // two S / P buffers
  static constexpr int Q_COL = 2 * kKT;
  static constexpr int O_COL = (D == 64) ? 192 : 256;
  static constexpr int TM_COLS = (O_COL + D <= 256) ? 256 : 512;
  static constexpr int NI = kKT * (D / 16) / kConv;  // 16-byte units per converter thread per tensor
};

enum Bar { K_FULL = 0, K_EMPTY = 3, V_FULL = 6, V_EMPTY = 9, S_FULL = 12, P_FULL = 14, PV_DONE = 16,
           Q_FULL = 17, FINAL = 18, NBAR = 19 };

// ------------------------------------------------------------ tcgen05 glue
// Shared-memory matrix descriptor: start address, leading / stride byte
// offsets (16-byte units), the fixed descriptor version 1 at bit 46 and the
// 128-byte swizzle mode (2) in bits 61-63.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor of kind::f16: FP32 accumulator (bits 4-5 = 1), f16 A
// and B (bits 7-12 = 0), B MN-major if b_mn (bit 16), N >> 3 in bits 17-22,
// M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, int b_mn) {
  return (1u << 4) | (static_cast<uint32_t>(b_mn) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               :: "r"(bar) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Non-blocking test of phase `parity` of a barrier (for polling several).
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}
// 32 lanes x 16 consecutive FP32 columns: thread t of the warp gets lane
// (32 * (warp % 4) + t) of the address's lane base.
__device__ __forceinline__ void tmem_ld16(uint32_t ta, uint32_t (&r)[16]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
               "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                 "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
               : "r"(ta));
}
__device__ __forceinline__ void tmem_st16(uint32_t ta, const uint32_t (&r)[16]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
               "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
               :: "r"(ta), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
                  "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]),
                  "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
               : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" :: "r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(p), "r"(bytes) : "memory");
}

// 16 E4M3 codes -> 8 f16x2 words, element order kept, exact.
__device__ __forceinline__ void e4m3x16_to_f16(const uint4 w, uint32_t (&o)[8]) {
  e4m3x4_to_f16x2x2(w.x, o[0], o[1]);
  e4m3x4_to_f16x2x2(w.y, o[2], o[3]);
  e4m3x4_to_f16x2x2(w.z, o[4], o[5]);
  e4m3x4_to_f16x2x2(w.w, o[6], o[7]);
}

// 32 lanes x 32 consecutive 32-bit columns (tcgen05.st).
__device__ __forceinline__ void tmem_st32(uint32_t ta, const uint32_t (&r)[32]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
               "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
               "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
               :: "r"(ta), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
                  "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
                  "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
                  "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
                  "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
               : "memory");
}
// O += A B with A in TMEM (f16 pairs, lane = row) and B from shared memory.
__device__ __forceinline__ void tc_mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
               :: "r"(d), "r"(a_tmem), "l"(b), "r"(id), "r"(acc) : "memory");
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t{1023});
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) extend_kernel(const ExtendArgs a) {
  using Gm = ExtGeo<D>;
  extern __shared__ uint8_t ext_raw[];
  __shared__ __align__(8) uint64_t bars[NBAR];
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int conv_tile;                 // tiles the converters have stored

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // this CTA's item (request b, query tile qt, head h) and key-range piece
  int item = blockIdx.x, piece = -1;                  // piece -1: the whole key range
  const int whole = a.items - a.split;
  if (item >= whole) {
    piece = (item - whole) % a.ways;
    item = whole + (item - whole) / a.ways;
  }
  const int h = item % a.Hq;
  const int qt = a.qtiles - 1 - (item / a.Hq) % a.qtiles;   // later query tiles (more keys) first
  const int b = item / (a.Hq * a.qtiles);
  const int C = a.chunk_lens[b], Lp = a.prefix_lens[b];
  if (qt == 0 && h == 0 && piece <= 0 && tid == 0 && (C < 0 || Lp < 0 || C > a.max_chunk_len))
    set_error(a.err, KV4_EBOUNDS);
  if (Lp < 0 || qt * kQT >= C) return;               // uniform over the CTA
  if (static_cast<int64_t>(Lp) + C >= (int64_t{1} << 31)) {
    if (tid == 0) set_error(a.err, KV4_EBOUNDS);
    return;
  }
  const int64_t c0 = a.cu_chunk[b], p0 = a.cu_prefix[b];
  const int rows = min(kQT, C - qt * kQT);
  const int kend = Lp + qt * kQT + rows;             // keys [0, kend) are visible to some row
  // Key tiles [jt0, jt0 + nT): all of them, or piece p of the full-prefix
  // tiles (every row sees all of those), the last piece taking the rest, so
  // no row's first tile in its piece is fully masked.
  int jt0 = 0, nT = (kend + kKT - 1) / kKT;
  if (piece >= 0) {
    const int np = Lp / kKT;
    const int j1 = (piece == a.ways - 1) ? nT : (piece + 1) * np / a.ways;
    jt0 = piece * np / a.ways;
    nT = j1 - jt0;
  }
  const int64_t pslot = static_cast<int64_t>(item - whole) * a.ways + piece;   // partial slot
  if (nT == 0) {
    // an empty piece: an empty state for the merge
    if (tid < kQT) reinterpret_cast<float2*>(a.part_ml)[pslot * kQT + tid] = make_float2(-INFINITY, 0.f);
    return;
  }
  const int hk = h / a.G;

  uint8_t* sm = align1024(ext_raw);
  const uint32_t sK = smem_u32(sm), sV = sK + Gm::OFF_V;
  const uint32_t bar0 = smem_u32(&bars[0]);
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };

  if (tid == 0) {
    for (int i = 0; i < kNST; ++i) {
      mbar_init(bar(K_FULL + i), kConv);
      mbar_init(bar(V_FULL + i), kConv);
      mbar_init(bar(K_EMPTY + i), 1);
      mbar_init(bar(V_EMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(S_FULL + i), 1);
      mbar_init(bar(P_FULL + i), 128);
    }
    mbar_init(bar(PV_DONE), 1);
    mbar_init(bar(Q_FULL), 128);
    mbar_init(bar(FINAL), 1);
    conv_tile = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(&tmem_slot)), "r"(Gm::TM_COLS) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t tO = tmem + Gm::O_COL, tQ = tmem + Gm::Q_COL;

  if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issue
    // One lane polls the operand barriers and issues whichever MMA is ready:
    // O += P_n V_n as soon as P_n and V_n are in; S_m = Q K_m^T (a whole
    // tile: issuing it in parts starves the tensor pipe) once K_m is in and
    // O += P_{m-2} V_{m-2}, the last reader of S buffer m % 2, has been issued.
    if (lane == 0) {
      bool ok = mbar_wait_bounded(bar(Q_FULL), 0);
      tc_fence_after();
      constexpr uint32_t idS = idesc_f16(kQT, kKT, 0), idO = idesc_f16(kQT, D, 1);
      int nS = 0, nP = 0, kst = 0, kph = 0, vst = 0, vph = 0;
      long long idle_since = clock64();
      while (ok && nP < nT) {
        bool progress = false;
        if (nP < nS && mbar_test(bar(P_FULL + (nP & 1)), (nP >> 1) & 1) &&
            mbar_test(bar(V_FULL + vst), vph)) {
          tc_fence_after();
          const uint64_t dV = sw128_desc(sV + vst * Gm::KV_BYTES, kKT * 128, 1024);
          const uint32_t tP = tmem + Gm::S_COL + (nP & 1) * kKT;
#pragma unroll
          for (int kk = 0; kk < kKT / 16; ++kk)
            tc_mma_ts(tO, tP + kk * 8, dV + ((kk * 2048) >> 4), idO, (nP > 0 || kk > 0));
#pragma unroll
          for (int kk = 0; kk < kKT / 16; ++kk)          // the lo part of P
            tc_mma_ts(tO, tP + 32 + kk * 8, dV + ((kk * 2048) >> 4), idO, 1);
          tc_commit(bar(PV_DONE));
          tc_commit(bar(V_EMPTY + vst));
          if (++vst == kNST) { vst = 0; vph ^= 1; }
          ++nP;
          progress = true;
        }
        if (nS < nT && (nS < 2 || nP >= nS - 1) && mbar_test(bar(K_FULL + kst), kph)) {
          tc_fence_after();
          const uint64_t dK = sw128_desc(sK + kst * Gm::KV_BYTES, 16, 1024);
          const uint32_t tS = tmem + Gm::S_COL + (nS & 1) * kKT;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ko = (kk >> 2) * (kKT * 128) + (kk & 3) * 32;
            tc_mma_ts(tS, tQ + kk * 8, dK + (ko >> 4), idS, kk > 0);
          }
          tc_commit(bar(S_FULL + (nS & 1)));
          tc_commit(bar(K_EMPTY + kst));
          if (++kst == kNST) { kst = 0; kph ^= 1; }
          ++nS;
          progress = true;
        }
        if (progress) {
          idle_since = clock64();
        } else if (clock64() - idle_since > kWaitCycles) {
          ok = false;
        }
      }
      if (!ok) set_error(a.err, KV4_ETIMEOUT);
      // Everything issued has completed once this arrives.
      tc_commit(bar(FINAL));
      if (!mbar_wait_bounded(bar(FINAL), 0)) set_error(a.err, KV4_ETIMEOUT);
    }
  } else if (warp == kPrefetchWarp) {
    // ------------------------------------------------------------ L2 prefetch
    // One bulk prefetch per tensor and tile over the tile's contiguous rows
    // (all kv heads: the CTAs of the other heads read them too), kept
    // kPrefetchAhead tiles ahead of the converters.
    if (lane == 0) {
      const int64_t rs = static_cast<int64_t>(a.Hkv) * D;
      auto prefetch = [&](int j) {
        const int k0 = (jt0 + j) * kKT, k1 = min(k0 + kKT, kend);
        const int e = min(k1, Lp), s0 = max(k0, Lp);
        if (k0 < e) {
          prefetch_l2(a.pk + (p0 + k0) * rs, static_cast<uint32_t>((e - k0) * rs));
          prefetch_l2(a.pv + (p0 + k0) * rs, static_cast<uint32_t>((e - k0) * rs));
        }
        if (s0 < k1) {
          prefetch_l2(a.ck + (c0 + s0 - Lp) * rs, static_cast<uint32_t>((k1 - s0) * rs));
          prefetch_l2(a.cv + (c0 + s0 - Lp) * rs, static_cast<uint32_t>((k1 - s0) * rs));
        }
      };
      int next = 1;
      long long idle_since = clock64();
      while (next < nT) {
        const int lim = min(nT, conv_tile + kPrefetchAhead);
        if (next < lim) {
          while (next < lim) prefetch(next++);
          idle_since = clock64();
        } else {
          __nanosleep(200);
          if (clock64() - idle_since > kWaitCycles) break;   // converters stopped: nothing to do
        }
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ converters
    constexpr int NI = Gm::NI, U16 = D / 16;
    const int t = tid - 128;
    const int64_t rs = static_cast<int64_t>(a.Hkv) * D;          // row stride (bytes)
    const uint8_t* pk = a.pk + (p0 * a.Hkv + hk) * static_cast<int64_t>(D);
    const uint8_t* pv = a.pv + (p0 * a.Hkv + hk) * static_cast<int64_t>(D);
    const uint8_t* ck = a.ck + (c0 * a.Hkv + hk) * static_cast<int64_t>(D);
    const uint8_t* cv = a.cv + (c0 * a.Hkv + hk) * static_cast<int64_t>(D);
    // Loads of one tensor's part of tile j into registers (zero past kend).
    auto load = [&](int j, const uint8_t* pre, const uint8_t* chk, uint4 (&w)[NI]) {
#pragma unroll
      for (int m = 0; m < NI; ++m) {
        const int it = m * kConv + t, r = it / U16, u = it % U16;
        const int key = (jt0 + j) * kKT + r;
        w[m] = make_uint4(0u, 0u, 0u, 0u);
        if (key < Lp) w[m] = __ldg(reinterpret_cast<const uint4*>(pre + key * rs) + u);
        else if (key < kend) w[m] = __ldg(reinterpret_cast<const uint4*>(chk + (key - Lp) * rs) + u);
      }
    };
    auto store = [&](uint32_t base, const uint4 (&w)[NI]) {
#pragma unroll
      for (int m = 0; m < NI; ++m) {
        const int it = m * kConv + t, r = it / U16, u = it % U16;
        uint32_t o[8];
        e4m3x16_to_f16(w[m], o);
        const int blk = u >> 2, c0u = (u & 3) * 2;
        const uint32_t row = base + blk * (kKT * 128) + r * 128;
        const int sw = r & 7, flip = blk & 1;     // alternate the unit order by column block
        const uint32_t a0 = row + (((c0u + flip) ^ sw) << 4);
        const uint32_t a1 = row + (((c0u + 1 - flip) ^ sw) << 4);
        if (flip) {
          sts128(a0, o[4], o[5], o[6], o[7]);
          sts128(a1, o[0], o[1], o[2], o[3]);
        } else {
          sts128(a0, o[0], o[1], o[2], o[3]);
          sts128(a1, o[4], o[5], o[6], o[7]);
        }
      }
    };
    // Stores of tile j's K (then V) into its stage, after the MMA that read
    // the stage's previous tile has completed.
    int kst = 0, kph = 0, vst = 0, vph = 0;
    auto put_k = [&](int j, const uint4 (&w)[NI]) -> bool {
      if (j >= kNST && !mbar_wait_bounded(bar(K_EMPTY + kst), kph ^ 1)) return false;
      store(sK + kst * Gm::KV_BYTES, w);
      fence_async_smem();
      mbar_arrive(bar(K_FULL + kst));
      if (++kst == kNST) { kst = 0; kph ^= 1; }
      return true;
    };
    auto put_v = [&](int j, const uint4 (&w)[NI]) -> bool {
      if (j >= kNST && !mbar_wait_bounded(bar(V_EMPTY + vst), vph ^ 1)) return false;
      store(sV + vst * Gm::KV_BYTES, w);
      fence_async_smem();
      mbar_arrive(bar(V_FULL + vst));
      if (++vst == kNST) { vst = 0; vph ^= 1; }
      if (t == 0) conv_tile = j + 1;
      return true;
    };
    // Two register sets, the loop unrolled by two: tile j+1's loads are in
    // flight while tile j is converted and stored.
    uint4 ak[NI], av[NI], bk[NI], bv[NI];
    load(0, pk, ck, ak);
    load(0, pv, cv, av);
    bool ok = true;
    for (int j = 0; j < nT; j += 2) {
      if (j + 1 < nT) {
        load(j + 1, pk, ck, bk);
        load(j + 1, pv, cv, bv);
      }
      if (!(ok = put_k(j, ak) && put_v(j, av)) || j + 1 >= nT) break;
      if (j + 2 < nT) {
        load(j + 2, pk, ck, ak);
        load(j + 2, pv, cv, av);
      }
      if (!(ok = put_k(j + 1, bk) && put_v(j + 1, bv))) break;
    }
    if (!ok && lane == 0) set_error(a.err, KV4_ETIMEOUT);
  } else {
    // ------------------------------------------------------------ softmax
    const int r = tid;                                // TMEM lane = query row
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    // Q row r: bf16 -> f16 pairs into TMEM (rows past the chunk are zero).
    {
      bool bad = false;
      const bool valid = r < rows;
      const uint4* src = reinterpret_cast<const uint4*>(
          a.q + ((c0 + qt * kQT + (valid ? r : 0)) * a.Hq + h) * static_cast<int64_t>(D));
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {              // 32 columns = 64 elements per store
        uint32_t v[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 w = valid ? __ldg(src + c * 8 + i) : make_uint4(0u, 0u, 0u, 0u);
          const uint32_t x[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float lo = __uint_as_float(x[k] << 16), hi = __uint_as_float(x[k] & 0xFFFF0000u);
            bad |= !(fabsf(lo) <= 65504.f) || !(fabsf(hi) <= 65504.f);
            v[4 * i + k] = pack_f16x2(lo, hi);
          }
        }
        tmem_st32(tQ + lane_base + c * 32, v);
      }
      tmem_wait_st();
      if (bad) set_error(a.err, KV4_EINVAL);
      tc_fence_before();
      mbar_arrive(bar(Q_FULL));
    }
    const float sk = a.fp8_scale[0], sv = a.fp8_scale[1];
    const float c2 = a.sm_scale * sk * kLog2e;           // S -> log2 units
    const int lim = min(Lp + qt * kQT + r, kend - 1);     // last key this row sees
    float m_use = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nT; ++j) {
      const int bb = j & 1;
      const uint32_t tS = tmem + Gm::S_COL + bb * kKT + lane_base;
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar(S_FULL + bb), (j >> 1) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[kKT];
#pragma unroll
      for (int c = 0; c < kKT / 16; ++c)
        tmem_ld16(tS + c * 16, *reinterpret_cast<uint32_t(*)[16]>(&sr[c * 16]));
      tmem_wait_ld();
      float s[kKT];
      const int kb = (jt0 + j) * kKT;
#pragma unroll
      for (int c = 0; c < kKT; ++c) s[c] = __uint_as_float(sr[c]);
      if (kb + kKT - 1 > lim) {
#pragma unroll
        for (int c = 0; c < kKT; ++c) s[c] = (kb + c <= lim) ? s[c] : -INFINITY;
      }
      float mx4[4] = {s[0], s[1], s[2], s[3]};        // four independent chains
#pragma unroll
      for (int c = 4; c < kKT; c += 4) {
#pragma unroll
        for (int i = 0; i < 4; ++i) mx4[i] = fmaxf(mx4[i], s[c + i]);
      }
      const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      const float mnew = mx * c2;
      const bool resc = mnew > m_use + 8.f;
      float alpha = 1.f;
      if (resc) {
        alpha = fast_exp2(m_use - mnew);
        m_use = mnew;
      }
      float rs4[4] = {0.f, 0.f, 0.f, 0.f};
      // P as an f16 hi + lo pair (about 22 significant bits): hi over the
      // first 32 columns of S_j, lo over the last 32
      uint32_t ph[kKT / 2], pl[kKT / 2];
#pragma unroll
      for (int c = 0; c < kKT; c += 2) {
        const float e0 = fast_exp2(fmaf(s[c], c2, -m_use));
        const float e1 = fast_exp2(fmaf(s[c + 1], c2, -m_use));
        rs4[(c >> 1) & 3] += e0 + e1;
        const uint32_t hi = pack_f16x2(e0, e1);
        const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hi));
        ph[c / 2] = hi;
        pl[c / 2] = pack_f16x2(e0 - hf.x, e1 - hf.y);
      }
      const float rs = (rs4[0] + rs4[1]) + (rs4[2] + rs4[3]);
      l = l * alpha + rs;
      if (j >= 1) {
        // O holds tiles < j once O += P_{j-1} V_{j-1} is done (waited every
        // tile to keep the barrier's phases in step; usually long complete)
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar(PV_DONE), (j - 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        // tcgen05.ld/st are warp-collective: the warp rescales when any of
        // its rows needs it (alpha is 1 for the others).
        if (__any_sync(0xffffffffu, resc)) {
#pragma unroll 1
          for (int c = 0; c < D / 16; ++c) {
            uint32_t o[16];
            tmem_ld16(tO + lane_base + c * 16, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st16(tO + lane_base + c * 16, o);
          }
        }
      }
      tmem_st32(tS, ph);                              // P_j over S_j: hi, then lo
      tmem_st32(tS + 32, pl);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(P_FULL + bb));
    }
    if (ok && !__all_sync(0xffffffffu, mbar_wait_bounded(bar(PV_DONE), (nT - 1) & 1))) ok = false;
    if (!ok) {
      if (lane == 0) set_error(a.err, KV4_ETIMEOUT);
    } else {
      tc_fence_after();
      const bool valid = r < rows;
      if (piece >= 0) {
        // a piece: its unnormalised O and (base, row sum) for the merge
        if (valid) reinterpret_cast<float2*>(a.part_ml)[pslot * kQT + r] = make_float2(m_use, l);
        float* po = a.part_o + (pslot * kQT + r) * static_cast<int64_t>(D);
#pragma unroll 1
        for (int c = 0; c < D / 16; ++c) {
          uint32_t o[16];
          tmem_ld16(tO + lane_base + c * 16, o);
          tmem_wait_ld();
          if (!valid) continue;
          float4* dst = reinterpret_cast<float4*>(po + c * 16);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_float4(__uint_as_float(o[4 * i]), __uint_as_float(o[4 * i + 1]),
                                 __uint_as_float(o[4 * i + 2]), __uint_as_float(o[4 * i + 3]));
        }
      }
      const float inv = sv / l;
      const int64_t orow = ((c0 + qt * kQT + r) * a.Hq + h) * static_cast<int64_t>(D);
#pragma unroll 1
      for (int c = 0; c < D / 16 && piece < 0; ++c) {
        uint32_t o[16];
        tmem_ld16(tO + lane_base + c * 16, o);
        tmem_wait_ld();
        if (!valid) continue;
        if (a.out_f32) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.out) + orow + c * 16);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv, __uint_as_float(o[4 * i + 1]) * inv,
                                 __uint_as_float(o[4 * i + 2]) * inv, __uint_as_float(o[4 * i + 3]) * inv);
        } else {
          uint32_t pk2[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const __nv_bfloat162 v2 = __floats2bfloat162_rn(__uint_as_float(o[2 * i]) * inv,
                                                            __uint_as_float(o[2 * i + 1]) * inv);
            pk2[i] = *reinterpret_cast<const uint32_t*>(&v2);
          }
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + orow + c * 16);
          dst[0] = make_uint4(pk2[0], pk2[1], pk2[2], pk2[3]);
          dst[1] = make_uint4(pk2[4], pk2[5], pk2[6], pk2[7]);
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                 :: "r"(tmem), "r"(Gm::TM_COLS) : "memory");
}

// Merge of the pieces of the split items: one warp per query row, the
// pieces' states in piece order (deterministic), O = sum_p 2^(m_p - M) O_p,
// l = sum_p 2^(m_p - M) l_p, out = O * s_V / l.
template <int D>
__global__ void __launch_bounds__(256) extend_merge_kernel(const ExtendArgs a) {
  const int k = blockIdx.x;
  const int item = a.items - a.split + k;
  const int h = item % a.Hq;
  const int qt = a.qtiles - 1 - (item / a.Hq) % a.qtiles;
  const int b = item / (a.Hq * a.qtiles);
  const int C = a.chunk_lens[b], Lp = a.prefix_lens[b];
  const int r = blockIdx.y * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (Lp < 0 || C < 0 || qt * kQT + r >= C || static_cast<int64_t>(Lp) + C >= (int64_t{1} << 31)) return;
  const float2* ml = reinterpret_cast<const float2*>(a.part_ml);
  float M = -INFINITY;
  for (int p = 0; p < a.ways; ++p) M = fmaxf(M, ml[(static_cast<int64_t>(k) * a.ways + p) * kQT + r].x);
  float l = 0.f;
  constexpr int NC = D / 128 > 0 ? D / 128 : 1;      // float4 columns per lane
  float4 acc[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int p = 0; p < a.ways; ++p) {
    const int64_t slot = static_cast<int64_t>(k) * a.ways + p;
    const float2 st = ml[slot * kQT + r];
    if (st.x == -INFINITY) continue;                 // an empty piece
    const float w = fast_exp2(st.x - M);
    l += w * st.y;
    const float4* po = reinterpret_cast<const float4*>(a.part_o + (slot * kQT + r) * D);
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int col = lane + 32 * c;
      if (col < D / 4) {
        const float4 v = __ldg(po + col);
        acc[c].x += w * v.x; acc[c].y += w * v.y; acc[c].z += w * v.z; acc[c].w += w * v.w;
      }
    }
  }
  const float inv = __ldg(a.fp8_scale + 1) / l;
  const int64_t orow = ((a.cu_chunk[b] + qt * kQT + r) * a.Hq + h) * static_cast<int64_t>(D);
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const int col = lane + 32 * c;
    if (col >= D / 4) continue;
    const float4 v = make_float4(acc[c].x * inv, acc[c].y * inv, acc[c].z * inv, acc[c].w * inv);
    if (a.out_f32) {
      reinterpret_cast<float4*>(static_cast<float*>(a.out) + orow)[col] = v;
    } else {
      const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
      reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + orow)[col] =
          make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
    }
  }
}

template <int D>
cudaError_t launch_d(const ExtendArgs& a, cudaStream_t st) {
  using Gm = ExtGeo<D>;
  // the shared-memory opt-in is per device; set it once per device (always
  // beyond the first 64 ids), racing threads set the same value
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(extend_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, Gm::SMEM);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  // one CTA per work-list entry: whole items, then the pieces of the split ones
  const int64_t ctas = static_cast<int64_t>(a.items - a.split) + static_cast<int64_t>(a.split) * a.ways;
  extend_kernel<D><<<static_cast<unsigned>(ctas), kThreads, Gm::SMEM, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || a.split == 0) return e;
  extend_merge_kernel<D><<<dim3(a.split, kQT / 8), 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

void extend_split(int items, int sms, int& split, int& ways) {
  // one CTA per SM (the kernel's shared memory): the items fill
  // floor(items / sms) waves and the remainder X a partial one; cutting the
  // remainder's key ranges into floor(sms / X) pieces spreads it over the SMs
  constexpr int kMaxWays = 16;
  split = 0;
  ways = 1;
  if (items <= 0 || sms <= 0) return;
  const int x = items >= sms ? items % sms : items;
  if (x == 0) return;
  const int w = sms / x < kMaxWays ? sms / x : kMaxWays;
  if (w < 2) return;
  split = x;
  ways = w;
}

cudaError_t launch_extend(const ExtendArgs& a, cudaStream_t st) {
  switch (a.D) {
    case 64: return launch_d<64>(a, st);
    case 128: return launch_d<128>(a, st);
    case 256: return launch_d<256>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kv4
