// Dequantise a cached 4-bit prefix into FP8 E4M3 workspaces: the first step
// of the chunked prefill / extend path of "SGLang's 4-bit KV cache", Figure 2,
// which turns the 4-bit prefix into FP8 in a buffer that is reused, then
// attends over prefix plus the current chunk.
//
// Every output byte is E4M3(RN(x_hat / s_fp8)) with RNE and saturation, where
// x_hat = RN((e2m1 * e4m3) * g) in FP32 (NVFP4) or RN(code * s) (INT4).  A
// 16-element block takes only a handful of distinct x_hat values (the eight
// E2M1 magnitudes under the block's E4M3 scale; the sixteen INT4 codes under
// the row's scale), so the kernel computes the output bytes of those values
// once, exactly as the per-element definition does, and turns each element
// into one byte selection from an 8-byte table (PRMT):
//
//  * NVFP4: the table depends only on the block-scale byte and the launch's
//    (g, s_fp8) of K or V, so each CTA builds all 256 of them (2 KB of shared
//    memory) once, with the IEEE division, and then streams.  E2M1 is
//    sign-magnitude and every step is odd in x, so a negative code takes its
//    magnitude's byte with the sign bit flipped.  (A NaN scale byte, which
//    the write never stores, gives a NaN byte of the code's sign where the
//    per-element computation would give 0x7F.)
//  * INT4: one FP32 scale per (token, head) row; each thread builds the two
//    tables of its row (codes 0..7 and 8..15 = -8..-1) with the correctly
//    rounded division on packed FP32 pairs.
//
// One thread converts 64 consecutive elements of one (token, head, K|V) row:
// 32 code bytes (64 for the token-pair rows of NVFP4 V, of which this token's
// nibbles are kept), one scale word, 64 bytes out.  One wave of resident
// CTAs strides over the rows, so the tables are built once per CTA; each
// thread loads its next item while it converts the current one, and a warp's
// 32 outputs (2 KB in a row of `out`) go out through shared memory as 512
// contiguous bytes a store instruction.
#include <cstdint>

#include "kv4_device.cuh"
#include "kv4_internal.h"

namespace kv4 {

constexpr int kPrefixThreads = 256;

__device__ __forceinline__ uint2 pack_e4m3x8(const float (&q)[8]) {
  return make_uint2(f32x2_to_e4m3x2(q[0], q[1]) | (f32x2_to_e4m3x2(q[2], q[3]) << 16),
                    f32x2_to_e4m3x2(q[4], q[5]) | (f32x2_to_e4m3x2(q[6], q[7]) << 16));
}

// NVFP4 table of scale byte sb: E4M3(RN(RN(e_i s g) / s8)) for the E2M1
// magnitudes e_i = 0, 0.5, 1, 1.5, 2, 3, 4, 6 (index = the code's low three
// bits).  e_i * s is exact in FP32 (at most 6 significant bits, within
// [2^-10, 2688]).
__device__ __forceinline__ uint2 nvfp4_scale_table(uint32_t sb, float g, float s8) {
  const float s = e4m3_to_f32(sb);
  const float e[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
  float q[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) q[i] = __fdiv_rn(__fmul_rn(__fmul_rn(e[i], s), g), s8);
  return pack_e4m3x8(q);
}

// The bytes of RN(x_i / s8) for 8 values x_i, as an 8-byte PRMT table.  Away
// from the FP32 range limits the division is div_rn on pairs, else the IEEE
// division.
__device__ __forceinline__ uint2 e4m3_table(const float (&x)[8], float s8, float r8, bool in_range) {
  float q[8];
  if (in_range) {
    const uint64_t nb = f2(-s8, -s8), yb2 = f2(r8, r8);
#pragma unroll
    for (int i = 0; i < 8; i += 2) div_rn_pair(x[i], x[i + 1], nb, yb2, q[i], q[i + 1]);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = __fdiv_rn(x[i], s8);
  }
  return pack_e4m3x8(q);
}

// Bit 0 of byte i = bit 3 of nibble i of sel (the code's sign), for the four
// low nibbles: PRMT from an all-0x80 table gives 0x80 for a selector below 8
// and the replicated sign bit, 0xFF, for one of 8 or more.
__device__ __forceinline__ uint32_t sign_bytes(uint32_t sel) { return prmt(0x80808080u, 0x80808080u, sel); }

// Four NVFP4 elements: mag_sel holds their codes' magnitude bits in its four
// low nibbles, signs has each element's sign in bit 7 of its byte (other bits
// ignored).
__device__ __forceinline__ uint32_t nvfp4_bytes(uint2 tab, uint32_t mag_sel, uint32_t signs) {
  return prmt(tab.x, tab.y, mag_sel) ^ (signs & 0x80808080u);
}

// Eight packed NVFP4 codes (element i in nibble i) -> 8 E4M3 bytes.
__device__ __forceinline__ uint2 nvfp4_word(uint2 tab, uint32_t w) {
  const uint32_t m = w & 0x77777777u;
  return make_uint2(nvfp4_bytes(tab, m, sign_bytes(w) << 7), nvfp4_bytes(tab, m >> 16, sign_bytes(w >> 16) << 7));
}

// Four NVFP4 elements of a token-pair row word x (element i in byte i, this
// token's nibble at bit sh of it) -> 4 E4M3 bytes.
__device__ __forceinline__ uint32_t nvfp4_pair_word(uint2 tab, uint32_t x, int sh) {
  const uint32_t xs = x >> sh;
  const uint32_t y = xs & 0x07070707u;
  const uint32_t sel = prmt(y | (y >> 4), 0u, 0x0020u);     // nibbles e0 e1 e2 e3
  return nvfp4_bytes(tab, sel, xs << 4);
}

// Eight INT4 codes (two's complement, element i in nibble i) -> 8 E4M3 bytes:
// tp holds the bytes of codes 0..7, tn those of 8..15.
__device__ __forceinline__ uint32_t int4_bytes(uint2 tp, uint2 tn, uint32_t mag_sel, uint32_t sel) {
  const uint32_t neg = prmt(sign_bytes(sel) << 7, 0u, 0xBA98u);   // 0xFF per negative code
  return (prmt(tp.x, tp.y, mag_sel) & ~neg) | (prmt(tn.x, tn.y, mag_sel) & neg);
}
__device__ __forceinline__ uint2 int4_word(uint2 tp, uint2 tn, uint32_t w) {
  const uint32_t m = w & 0x77777777u;
  return make_uint2(int4_bytes(tp, tn, m, w), int4_bytes(tp, tn, m >> 16, w >> 16));
}

// A warp's 32 items are 32 consecutive 64-byte pieces of the output.  Each
// lane puts its 64 bytes (chunks L = 4 lane + j of 16 bytes) in one of the
// warp's two 2 KB buffers, chunk L at row L / 8, column (L % 8) ^ (row % 8)
// of 128-byte rows: the 128-byte swizzle of the tensor copy unit, and free of
// bank conflicts both ways.  Then one lane stores the 2 KB with a tensor copy
// through `tmap` (the output viewed as 128-byte rows, row `y`), or, for a step
// with items to skip or a start off a 128-byte boundary, lane l stores
// linear chunks 32 m + l (m = 0..3) itself, 512 contiguous bytes an
// instruction.  `valid` holds bit k for each item k of the 32 to be written.
// Every step commits one bulk group; a buffer is refilled only after the
// group that read it two steps before has finished reading.
__device__ __forceinline__ uint32_t tchunk(uint32_t L) { return L ^ ((L >> 3) & 7u); }

__device__ __forceinline__ void store_warp(uint4* gdst, uint32_t sbuf, uint32_t lane, const uint4 (&o)[4],
                                           uint32_t valid, const CUtensorMap* tmap, int64_t y) {
  if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
  __syncwarp();
  if (valid >> lane & 1u) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t addr = sbuf + 16 * tchunk(4 * lane + j);
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(o[j].x), "r"(o[j].y), "r"(o[j].z),
                   "r"(o[j].w)
                   : "memory");
    }
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // visible to the tensor copy
  __syncwarp();
  if (valid == 0xFFFFFFFFu && y >= 0) {
    if (lane == 0)
      asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
                   ::"l"(reinterpret_cast<uint64_t>(tmap)), "r"(0), "r"(static_cast<int>(y)), "r"(sbuf)
                   : "memory");
  } else {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const uint32_t L = 32 * m + lane;
      if (valid >> (L >> 2) & 1u) gdst[L] = lds128(sbuf + 16 * tchunk(L));
    }
  }
  if (lane == 0) asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// The walk of one (kind, request) CTA over its items (kind K|V = 0|1).
template <int D, int FMT, int kind>
__device__ __forceinline__ void prefix_walk(const PrefixArgs& a, uint32_t items, int64_t obase, const int32_t* table,
                                            uint8_t* out, float s8, const uint2* s_tab, uint8_t* s_out,
                                            const CUtensorMap* tmap) {
  constexpr int TPR = D / 64;                   // threads per row
  constexpr int RB = D / 2, SB = D / 16;
  constexpr bool VP = FMT == KV4_NVFP4 && kind == 1;   // NVFP4 V: token-pair rows
  constexpr bool VP16 = FMT == KV4_INT4_PTH && kind == 1;   // INT4 V: pair rows by 16-bit halves
  const float r8 = __frcp_rn(s8);
  // Two-deep software pipeline: the next item's block-table entry and code
  // loads are in flight while this item is converted and stored.
  struct Item {
    uint4 c[VP || VP16 ? 4 : 2]; // codes: 32 bytes, or the 64 of a V pair-row span
    uint2 sw;            // scale bytes (NVFP4) or the row scale's bits (INT4, in .x)
    int sh;              // V pair rows: this token's place in the pair (off % 2)
    bool ok;             // false: nothing to do
  };
  auto load = [&](uint32_t i, Item& it) {
    it.ok = false;
    if (i >= items) return;
    const uint32_t row = i / TPR;
    const int part = static_cast<int>(i % TPR);
    const uint32_t t = fdiv(row, a.hkv_div);
    const int h = static_cast<int>(row - t * static_cast<uint32_t>(a.Hkv));
    const uint32_t pidx = fdiv(t, a.p_div);
    const int page = __ldg(table + pidx);
    if (page < 0 || page >= a.num_pages) {
      if (part == 0) set_error(a.err, KV4_EBOUNDS);
      return;
    }
    const int off = static_cast<int>(t - pidx * static_cast<uint32_t>(a.P));
    const uint8_t* chunk = a.pool + (static_cast<int64_t>(page) * a.Hkv + h) * a.chunk_bytes;
    it.ok = true;
    if constexpr (VP) {
      // V is stored in token pairs: byte d of pair row off/2 holds element d
      // of this token in nibble off%2; scale byte 2 blk + off%2 of the pair
      const uint4* src = reinterpret_cast<const uint4*>(
          chunk + static_cast<int64_t>(a.P) * RB + static_cast<int64_t>(off >> 1) * D + part * 64);
#pragma unroll
      for (int j = 0; j < 4; ++j) it.c[j] = src[j];
      it.sw = *reinterpret_cast<const uint2*>(chunk + static_cast<int64_t>(a.P) * D + static_cast<int64_t>(a.P) * SB +
                                              static_cast<int64_t>(off >> 1) * 2 * SB + part * 8);
      it.sh = off & 1;
    } else if constexpr (VP16) {
      // INT4 V in token pairs: word k of pair row off/2 holds the token's
      // 16-bit chunk k in its half off%2; the row scale stays per token
      const uint4* src = reinterpret_cast<const uint4*>(
          chunk + static_cast<int64_t>(a.P) * RB + static_cast<int64_t>(off >> 1) * D + part * 64);
#pragma unroll
      for (int j = 0; j < 4; ++j) it.c[j] = src[j];
      it.sw.x = *reinterpret_cast<const uint32_t*>(chunk + static_cast<int64_t>(a.P) * D +
                                                   (static_cast<int64_t>(a.P) + off) * 4);
      it.sh = off & 1;
    } else {
      const uint4* src = reinterpret_cast<const uint4*>(chunk + static_cast<int64_t>(kind) * a.P * RB +
                                                        static_cast<int64_t>(off) * RB + part * 32);
      it.c[0] = src[0];
      it.c[1] = src[1];
      if constexpr (FMT == KV4_NVFP4) {
        // the four blocks' scale bytes, in order
        it.sw.x = *reinterpret_cast<const uint32_t*>(chunk + static_cast<int64_t>(a.P) * D +
                                                     static_cast<int64_t>(off) * SB + part * 4);
      } else {
        it.sw.x = *reinterpret_cast<const uint32_t*>(chunk + static_cast<int64_t>(a.P) * D +
                                                     (static_cast<int64_t>(kind) * a.P + off) * 4);
      }
    }
  };

  const uint32_t stride = gridDim.x * kPrefixThreads;
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t sbuf0 = smem_u32(s_out) + (threadIdx.x >> 5) * 4096u;   // the warp's two buffers
  uint4* gout = reinterpret_cast<uint4*>(out + obase * a.Hkv * D);
  // the request's first output byte in 128-byte rows of the tensor view, or
  // -1 when it is off a row boundary (then every step stores from the lanes)
  const int64_t obyte = obase * a.Hkv * D;
  const int64_t yrow = (obyte % 128 == 0) ? obyte / 128 : -1;
  uint32_t buf = 0;
  Item cur, nxt;
  // warp-uniform walk: the warp's items are ib + lane
  uint32_t ib = blockIdx.x * kPrefixThreads + (threadIdx.x & ~31u);
  load(ib + lane, cur);
  for (; ib < items; ib += stride) {
    load(ib + stride + lane, nxt);
    uint4 o[4];
    if (cur.ok) {
      if constexpr (FMT == KV4_NVFP4) {
        if constexpr (!VP) {
          const uint32_t cw[8] = {cur.c[0].x, cur.c[0].y, cur.c[0].z, cur.c[0].w,
                                  cur.c[1].x, cur.c[1].y, cur.c[1].z, cur.c[1].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint2 tab = s_tab[(cur.sw.x >> (8 * j)) & 0xFFu];
            const uint2 lo = nvfp4_word(tab, cw[2 * j]), hi = nvfp4_word(tab, cw[2 * j + 1]);
            o[j] = make_uint4(lo.x, lo.y, hi.x, hi.y);
          }
        } else {
          const int sh = 4 * cur.sh;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t sbw = j < 2 ? cur.sw.x : cur.sw.y;
            const uint2 tab = s_tab[(sbw >> (16 * (j & 1) + 8 * cur.sh)) & 0xFFu];
            const uint4 x = cur.c[j];
            o[j] = make_uint4(nvfp4_pair_word(tab, x.x, sh), nvfp4_pair_word(tab, x.y, sh),
                              nvfp4_pair_word(tab, x.z, sh), nvfp4_pair_word(tab, x.w, sh));
          }
        }
      } else {
        const float s = __uint_as_float(cur.sw.x);
        // the row's tables: codes 0..7 and 8..15 (values -8..-1), x = RN(code * s)
        const bool in_range = div_rn_in_range(r8, 16.f * fabsf(s));
        const uint64_t ss = f2(s, s);
        float xp[8], xn[8];
#pragma unroll
        for (int k = 0; k < 8; k += 2) {
          f2_split(mul_f2(f2(static_cast<float>(k), static_cast<float>(k + 1)), ss), xp[k], xp[k + 1]);
          f2_split(mul_f2(f2(static_cast<float>(k - 8), static_cast<float>(k - 7)), ss), xn[k], xn[k + 1]);
        }
        const uint2 tp = e4m3_table(xp, s8, r8, in_range), tn = e4m3_table(xn, s8, r8, in_range);
        uint32_t cw[8];
        if constexpr (VP16) {
          // the token's code words back from its halves of the pair words
          const uint32_t sel = cur.sh ? 0x7632u : 0x5410u;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            cw[2 * j] = prmt(cur.c[j].x, cur.c[j].y, sel);
            cw[2 * j + 1] = prmt(cur.c[j].z, cur.c[j].w, sel);
          }
        } else {
          const uint32_t c8[8] = {cur.c[0].x, cur.c[0].y, cur.c[0].z, cur.c[0].w,
                                  cur.c[1].x, cur.c[1].y, cur.c[1].z, cur.c[1].w};
#pragma unroll
          for (int j = 0; j < 8; ++j) cw[j] = c8[j];
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint2 lo = int4_word(tp, tn, cw[2 * j]), hi = int4_word(tp, tn, cw[2 * j + 1]);
          o[j] = make_uint4(lo.x, lo.y, hi.x, hi.y);
        }
      }
    }
    const int64_t y = yrow < 0 ? -1 : yrow + static_cast<int64_t>(ib) / 2;     // 64 ib bytes = ib / 2 rows
    store_warp(gout + 4 * static_cast<int64_t>(ib), sbuf0 + 2048u * buf, lane, o, __ballot_sync(0xFFFFFFFFu, cur.ok),
               tmap, y < (int64_t{1} << 31) - 16 ? y : -1);
    buf ^= 1u;
    cur = nxt;
  }
  if ((threadIdx.x & 31u) == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// CTA (gx, kind = blockIdx.y, request b = blockIdx.z); item i of request b =
// (row = (t, h), part): elements [64 part, 64 part + 64) of that row.
template <int D, int FMT>
__global__ void __launch_bounds__(kPrefixThreads, 3)
prefix_kernel(const PrefixArgs a, const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v) {
  constexpr int TPR = D / 64;                   // threads per row
  __shared__ uint2 s_tab[FMT == KV4_NVFP4 ? 256 : 1];
  __shared__ __align__(1024) uint8_t s_out[(kPrefixThreads / 32) * 4096];   // per warp: two 2 KB buffers
  const int b = blockIdx.z;
  const int kind = blockIdx.y;
  const float s8 = __ldg(a.fp8_scale + kind);
  if constexpr (FMT == KV4_NVFP4) {
    s_tab[threadIdx.x] = nvfp4_scale_table(threadIdx.x, __ldg(a.gscale + kind), s8);
    __syncthreads();
  }
  int n = a.prefix_lens[b];
  const int cap = min(a.max_prefix_len, a.max_pages * a.P);
  if (n < 0 || n > cap) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_error(a.err, KV4_EBOUNDS);
    n = n < 0 ? 0 : cap;
  }
  const uint32_t items = static_cast<uint32_t>(n) * static_cast<uint32_t>(a.Hkv) * TPR;
  const int64_t obase = a.cu_prefix[b];
  const int32_t* table = a.block_table + static_cast<int64_t>(b) * a.max_pages;
  uint8_t* out = kind == 0 ? a.out_k : a.out_v;
  if (kind == 0) prefix_walk<D, FMT, 0>(a, items, obase, table, out, s8, s_tab, s_out, &map_k);
  else prefix_walk<D, FMT, 1>(a, items, obase, table, out, s8, s_tab, s_out, &map_v);
}

template <int D, int FMT>
static cudaError_t launch_prefix_t(const PrefixArgs& a, const CUtensorMap& mk, const CUtensorMap& mv, cudaStream_t st) {
  const int64_t items = static_cast<int64_t>(a.max_prefix_len) * a.Hkv * (D / 64);
  const int64_t need = (items + kPrefixThreads - 1) / kPrefixThreads;
  // one wave of resident CTAs over all (kind, request) pairs; each strides
  // over its request's rows
  static int per_sm = 0;
  if (per_sm == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, prefix_kernel<D, FMT>, kPrefixThreads, 0) !=
            cudaSuccess || n < 1)
      n = 4;
    per_sm = n;
  }
  const int64_t target = (static_cast<int64_t>(a.sms) * per_sm + 2 * a.B - 1) / (2 * a.B);
  const int64_t gx = need < target ? need : (target > 0 ? target : 1);
  prefix_kernel<D, FMT><<<dim3(static_cast<unsigned>(gx), 2, a.B), kPrefixThreads, 0, st>>>(a, mk, mv);
  return cudaGetLastError();
}

cudaError_t launch_prefix(const PrefixArgs& a_in, const CUtensorMap& mk, const CUtensorMap& mv, cudaStream_t st) {
  if (a_in.max_prefix_len == 0 || a_in.B == 0) return cudaSuccess;
  PrefixArgs a = a_in;
  a.hkv_div = make_fastdiv(static_cast<uint32_t>(a.Hkv));
  a.p_div = make_fastdiv(static_cast<uint32_t>(a.P));
  if (a.fmt == KV4_NVFP4) {
    switch (a.D) {
      case 64: return launch_prefix_t<64, KV4_NVFP4>(a, mk, mv, st);
      case 128: return launch_prefix_t<128, KV4_NVFP4>(a, mk, mv, st);
      default: return launch_prefix_t<256, KV4_NVFP4>(a, mk, mv, st);
    }
  }
  switch (a.D) {
    case 64: return launch_prefix_t<64, KV4_INT4_PTH>(a, mk, mv, st);
    case 128: return launch_prefix_t<128, KV4_INT4_PTH>(a, mk, mv, st);
    default: return launch_prefix_t<256, KV4_INT4_PTH>(a, mk, mv, st);
  }
}

}  // namespace kv4
