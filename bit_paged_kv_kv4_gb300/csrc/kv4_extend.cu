// Chunked-prefill / extend attention over the FP8 workspace plus the FP8
// current chunk ("SGLang's 4-bit KV cache", Figure 2, right-hand column: the
// cached prefix is dequantised into a reused FP8 workspace and the chunk's
// queries attend over prefix plus current chunk).  Chunk query i of a
// request sits at position Lp + i and sees all Lp prefix keys and the chunk
// keys 0..i.  One per-tensor FP8 scale pair {s_K, s_V} serves both.
//
// This is the dense part of the path, so it runs on the fifth-generation
// tensor cores: tcgen05.mma kind::f16 with the accumulators in tensor memory.
// One CTA owns 128 query rows of one query head (the MMA's M) and streams the
// request's keys in tiles of 64:
//
//   warps 0-3   softmax, one thread per query row: S from TMEM, mask, online
//               softmax in the log2 domain, P (f16) into shared memory, the
//               rare rescale of O in TMEM, and the epilogue.
//   warps 4-7   converters: FP8 K and V rows from global memory (one tile in
//               registers ahead, three tiles ahead into L2) to f16 tiles in
//               the 128-byte-swizzled layout the MMA reads.
//   warp 8      TMEM allocation and, on one lane, the MMA issue:
//               S_j = Q K_j^T (M128 N64, K = head_dim), then O += P_{j-1} V_{j-1}
//               (M128 N=head_dim K64), so S_j overlaps the softmax of tile j-1.
//
// Operand layouts (all K-major rows of 128 bytes, 8-row swizzle atoms of 1024
// bytes, 16-byte unit index XOR row % 8):
//   Q  f16 [D/64][128 rows][64]        A of S   (stride between 8-row groups 1024)
//   K  f16 [D/64][64 keys][64]         B of S   (K-major)
//   P  f16 [128 rows][64 keys]         A of O
//   V  f16 [D/64][64 keys][64]         B of O, MN-major: N = head_dim runs along
//                                      the 128-byte rows; 64-column blocks are
//                                      the leading-byte-offset stride (64*128),
//                                      8-key groups the stride-byte-offset (1024)
//
// Exact FP8 -> f16 by integer ops: with the E4M3 byte b placed in a 16-bit
// lane, (b + (b & 0x80)) << 7 is the f16 whose value is e4m3(b) * 2^-8, for
// normal and subnormal codes alike (f16 exponent bias 15 = 7 + 8).  The 2^8
// is folded into the softmax scale for K and the output scale for V.  Q is
// converted bf16 -> f16 once per CTA (exact for 2^-14 <= |q| <= 65504; larger
// magnitudes are flagged).  P is rounded to f16 once (relative 2^-11); S and
// O accumulate in FP32.
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
constexpr int kThreads = 288;     // 4 softmax warps, 4 converter warps, 1 MMA warp
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct ExtGeo {
  static constexpr int Q_BYTES = kQT * D * 2;
  static constexpr int KV_BYTES = kKT * D * 2;
  static constexpr int P_BYTES = kQT * kKT * 2;
  static constexpr int OFF_K = Q_BYTES;          // two buffers
  static constexpr int OFF_V = OFF_K + 2 * KV_BYTES;
  static constexpr int OFF_P = OFF_V + 2 * KV_BYTES;
  static constexpr int SMEM = OFF_P + P_BYTES + 1024;   // + alignment slack
  static constexpr int TM_COLS = (2 * kKT + D <= 256) ? 256 : 512;
  static constexpr int O_COL = TM_COLS / 2;      // S buffers at columns 0 and 64
  static constexpr int NI = kKT * (D / 16) / 128;  // 16-byte units per converter thread per tensor
};

enum Bar { KV_FULL = 0, KV_EMPTY = 2, S_FULL = 4, S_EMPTY = 6, P_FULL = 8, PV_DONE = 9, FINAL = 10,
           NBAR = 11 };

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
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
               :: "r"(d), "l"(a), "l"(b), "r"(id), "r"(acc) : "memory");
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

// Two E4M3 bytes in the low bytes of 16-bit lanes -> f16x2 of value * 2^-8.
__device__ __forceinline__ uint32_t e4m3_lanes_to_f16x2(uint32_t y) {
  return (y + (y & 0x00800080u)) << 7;
}
// 16 E4M3 codes -> 8 f16x2 words (value * 2^-8), element order kept.
__device__ __forceinline__ void e4m3x16_to_f16(const uint4 w, uint32_t (&o)[8]) {
  const uint32_t x[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    o[2 * i] = e4m3_lanes_to_f16x2(prmt(x[i], 0u, 0x4140u));
    o[2 * i + 1] = e4m3_lanes_to_f16x2(prmt(x[i], 0u, 0x4342u));
  }
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

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x, qt = blockIdx.y, b = blockIdx.z;
  const int C = a.chunk_lens[b], Lp = a.prefix_lens[b];
  if (qt == 0 && h == 0 && tid == 0 && (C < 0 || Lp < 0 || C > a.max_chunk_len))
    set_error(a.err, KV4_EBOUNDS);
  if (Lp < 0 || qt * kQT >= C) return;               // uniform over the CTA
  if (static_cast<int64_t>(Lp) + C >= (int64_t{1} << 31)) {
    if (tid == 0) set_error(a.err, KV4_EBOUNDS);
    return;
  }
  const int64_t c0 = a.cu_chunk[b], p0 = a.cu_prefix[b];
  const int rows = min(kQT, C - qt * kQT);
  const int kend = Lp + qt * kQT + rows;             // keys [0, kend) are visible to some row
  const int nT = (kend + kKT - 1) / kKT;
  const int hk = h / a.G;

  uint8_t* sm = align1024(ext_raw);
  const uint32_t sQ = smem_u32(sm), sK = sQ + Gm::OFF_K, sV = sQ + Gm::OFF_V, sP = sQ + Gm::OFF_P;
  const uint32_t bar0 = smem_u32(&bars[0]);
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };

  if (tid == 0) {
    mbar_init(bar(KV_FULL), 128);
    mbar_init(bar(KV_FULL + 1), 128);
    mbar_init(bar(KV_EMPTY), 1);
    mbar_init(bar(KV_EMPTY + 1), 1);
    mbar_init(bar(S_FULL), 1);
    mbar_init(bar(S_FULL + 1), 1);
    mbar_init(bar(S_EMPTY), 128);
    mbar_init(bar(S_EMPTY + 1), 128);
    mbar_init(bar(P_FULL), 128);
    mbar_init(bar(PV_DONE), 1);
    mbar_init(bar(FINAL), 1);
    fence_mbar_init();
  }
  if (warp == 8) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(&tmem_slot)), "r"(Gm::TM_COLS) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }

  // Q rows of this CTA: bf16 -> f16 into the swizzled A layout (rows past
  // the chunk are zero).  Warps 0-7, one 16-byte unit per thread and step.
  bool bad = false;
  if (tid < 256) {
    constexpr int U = D / 8;                          // 16-byte units per row
    for (int it = tid; it < kQT * U; it += 256) {
      const int r = it / U, u = it % U;
      uint4 w = make_uint4(0u, 0u, 0u, 0u);
      if (r < rows) {
        const __nv_bfloat16* src = a.q + ((c0 + qt * kQT + r) * a.Hq + h) * static_cast<int64_t>(D) + u * 8;
        w = __ldg(reinterpret_cast<const uint4*>(src));
      }
      uint32_t x[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float lo = __uint_as_float(x[i] << 16), hi = __uint_as_float(x[i] & 0xFFFF0000u);
        bad |= !(fabsf(lo) <= 65504.f) || !(fabsf(hi) <= 65504.f);
        x[i] = pack_f16x2(lo, hi);
      }
      const uint32_t addr = sQ + (u >> 3) * (kQT * 128) + r * 128 + (((u & 7) ^ (r & 7)) << 4);
      sts128(addr, x[0], x[1], x[2], x[3]);
    }
    fence_async_smem();
  }
  tc_fence_before();
  const int any_bad = __syncthreads_or(bad);
  tc_fence_after();
  if (any_bad && tid == 0) set_error(a.err, KV4_EINVAL);
  const uint32_t tmem = tmem_slot;
  const uint32_t tO = tmem + Gm::O_COL;

  if (warp == 8) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      bool ok = true;
      constexpr uint32_t idS = idesc_f16(kQT, kKT, 0), idO = idesc_f16(kQT, D, 1);
      const uint64_t dQ = sw128_desc(sQ, 16, 1024);
      for (int j = 0; j <= nT && ok; ++j) {
        if (j < nT) {
          const int bb = j & 1;
          ok = mbar_wait_bounded(bar(KV_FULL + bb), (j >> 1) & 1) &&
               (j < 2 || mbar_wait_bounded(bar(S_EMPTY + bb), ((j - 2) >> 1) & 1));
          if (!ok) break;
          tc_fence_after();
          const uint64_t dK = sw128_desc(sK + bb * Gm::KV_BYTES, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t qo = (kk >> 2) * (kQT * 128) + (kk & 3) * 32;
            const uint32_t ko = (kk >> 2) * (kKT * 128) + (kk & 3) * 32;
            tc_mma(tmem + bb * kKT, dQ + (qo >> 4), dK + (ko >> 4), idS, kk > 0);
          }
          tc_commit(bar(S_FULL + bb));
        }
        if (j >= 1) {
          const int jp = j - 1, pb = jp & 1;
          ok = mbar_wait_bounded(bar(P_FULL), jp & 1);
          if (!ok) break;
          tc_fence_after();
          const uint64_t dP = sw128_desc(sP, 16, 1024);
          const uint64_t dV = sw128_desc(sV + pb * Gm::KV_BYTES, kKT * 128, 1024);
#pragma unroll
          for (int kk = 0; kk < kKT / 16; ++kk)
            tc_mma(tO, dP + ((kk * 32) >> 4), dV + ((kk * 2048) >> 4), idO, (jp > 0 || kk > 0));
          tc_commit(bar(PV_DONE));
          tc_commit(bar(KV_EMPTY + pb));
        }
      }
      if (!ok) set_error(a.err, KV4_ETIMEOUT);
      // Everything issued has completed once this arrives.
      tc_commit(bar(FINAL));
      if (!mbar_wait_bounded(bar(FINAL), 0)) set_error(a.err, KV4_ETIMEOUT);
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
    auto load = [&](int j, uint4 (&kr)[NI], uint4 (&vr)[NI]) {
#pragma unroll
      for (int m = 0; m < NI; ++m) {
        const int it = m * 128 + t, r = it / U16, u = it % U16;
        const int key = j * kKT + r;
        kr[m] = make_uint4(0u, 0u, 0u, 0u);
        vr[m] = kr[m];
        if (key < Lp) {
          kr[m] = __ldg(reinterpret_cast<const uint4*>(pk + key * rs) + u);
          vr[m] = __ldg(reinterpret_cast<const uint4*>(pv + key * rs) + u);
        } else if (key < kend) {
          kr[m] = __ldg(reinterpret_cast<const uint4*>(ck + (key - Lp) * rs) + u);
          vr[m] = __ldg(reinterpret_cast<const uint4*>(cv + (key - Lp) * rs) + u);
        }
      }
    };
    auto prefetch = [&](int j) {
      if (j >= nT) return;
      const int key = j * kKT + (t & 63);
      const bool isv = t >= 64;
      if (key < Lp) prefetch_l2((isv ? pv : pk) + key * rs, D);
      else if (key < kend) prefetch_l2((isv ? cv : ck) + (key - Lp) * rs, D);
    };
    auto store = [&](uint32_t base, const uint4 (&w)[NI]) {
#pragma unroll
      for (int m = 0; m < NI; ++m) {
        const int it = m * 128 + t, r = it / U16, u = it % U16;
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
    uint4 kc[NI], vc[NI];
    prefetch(1);
    prefetch(2);
    load(0, kc, vc);
    bool ok = true;
    for (int j = 0; j < nT; ++j) {
      const int bb = j & 1;
      uint4 kn[NI], vn[NI];
      prefetch(j + 3);
      if (j + 1 < nT) load(j + 1, kn, vn);
      if (j >= 2 && !mbar_wait_bounded(bar(KV_EMPTY + bb), ((j - 2) >> 1) & 1)) { ok = false; break; }
      store(sK + bb * Gm::KV_BYTES, kc);
      store(sV + bb * Gm::KV_BYTES, vc);
      fence_async_smem();
      mbar_arrive(bar(KV_FULL + bb));
#pragma unroll
      for (int m = 0; m < NI; ++m) { kc[m] = kn[m]; vc[m] = vn[m]; }
    }
    if (!ok && lane == 0) set_error(a.err, KV4_ETIMEOUT);
  } else {
    // ------------------------------------------------------------ softmax
    const int r = tid;                                // TMEM lane = query row
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const float sk = a.fp8_scale[0], sv = a.fp8_scale[1];
    const float c2 = a.sm_scale * sk * 256.f * kLog2e;   // S from the 2^-8 operands -> log2 units
    const int lim = min(Lp + qt * kQT + r, kend - 1);     // last key this row sees
    float m_use = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nT; ++j) {
      const int bb = j & 1;
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar(S_FULL + bb), (j >> 1) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[kKT];
#pragma unroll
      for (int c = 0; c < kKT / 16; ++c)
        tmem_ld16(tmem + lane_base + bb * kKT + c * 16, *reinterpret_cast<uint32_t(*)[16]>(&sr[c * 16]));
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(bar(S_EMPTY + bb));
      float s[kKT];
      const int kb = j * kKT;
#pragma unroll
      for (int c = 0; c < kKT; ++c) s[c] = __uint_as_float(sr[c]);
      if (kb + kKT - 1 > lim) {
#pragma unroll
        for (int c = 0; c < kKT; ++c) s[c] = (kb + c <= lim) ? s[c] : -INFINITY;
      }
      float mx = s[0];
#pragma unroll
      for (int c = 1; c < kKT; ++c) mx = fmaxf(mx, s[c]);
      const float mnew = mx * c2;
      const bool resc = mnew > m_use + 8.f;
      float alpha = 1.f;
      if (resc) {
        alpha = fast_exp2(m_use - mnew);
        m_use = mnew;
      }
      float rs = 0.f;
      uint32_t ph[kKT / 2];
#pragma unroll
      for (int c = 0; c < kKT; c += 2) {
        const float e0 = fast_exp2(fmaf(s[c], c2, -m_use));
        const float e1 = fast_exp2(fmaf(s[c + 1], c2, -m_use));
        rs += e0 + e1;
        ph[c / 2] = pack_f16x2(e0, e1);
      }
      l = l * alpha + rs;
      if (j >= 1) {
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
          tmem_wait_st();
        }
      }
#pragma unroll
      for (int c = 0; c < 8; ++c)
        sts128(sP + r * 128 + ((c ^ (r & 7)) << 4), ph[4 * c], ph[4 * c + 1], ph[4 * c + 2], ph[4 * c + 3]);
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(bar(P_FULL));
    }
    if (ok && !__all_sync(0xffffffffu, mbar_wait_bounded(bar(PV_DONE), (nT - 1) & 1))) ok = false;
    if (!ok) {
      if (lane == 0) set_error(a.err, KV4_ETIMEOUT);
    } else {
      tc_fence_after();
      const bool valid = r < rows;
      const float inv = sv * 256.f / l;
      const int64_t orow = ((c0 + qt * kQT + r) * a.Hq + h) * static_cast<int64_t>(D);
#pragma unroll 1
      for (int c = 0; c < D / 16; ++c) {
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
  if (warp == 8)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                 :: "r"(tmem), "r"(Gm::TM_COLS) : "memory");
}

template <int D>
cudaError_t launch_d(const ExtendArgs& a, cudaStream_t st) {
  using Gm = ExtGeo<D>;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(extend_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, Gm::SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const dim3 grid(a.Hq, (a.max_chunk_len + kQT - 1) / kQT, a.B);
  extend_kernel<D><<<grid, kThreads, Gm::SMEM, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_extend(const ExtendArgs& a, cudaStream_t st) {
  switch (a.D) {
    case 64: return launch_d<64>(a, st);
    case 128: return launch_d<128>(a, st);
    case 256: return launch_d<256>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kv4
