// The C ABI of libkv4 (declared in include/kv4.h): host-side validation,
// workspace sizing, TMA descriptor set-up and dispatch to the kernels.
//
// Every entry point validates its arguments before touching the CUDA
// runtime, so argument errors are reported (and testable) on machines without
// a GPU.  Nothing here allocates device memory or synchronises the host,
// except kv4_device_error(), which reads the per-device error word.
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/kv4.h"
#include "kv4_internal.h"

namespace {

thread_local std::string g_msg;

kv4_status fail(kv4_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_msg = buf;
  return s;
}

kv4_status cuda_fail(cudaError_t e, const char* what) {
  return fail(KV4_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int64_t chunk_bytes_of(const kv4_pool& p) {
  const int64_t P = p.page_size, D = p.head_dim;
  return p.fmt == KV4_NVFP4 ? P * (D + D / 8)
         : p.fmt == KV4_FP8   ? P * 2 * D
         : p.fmt == KV4_K8V4  ? P * (D + D / 2 + 4)
                              : P * (D + 8);
}

kv4_status check_pool(const kv4_pool* p) {
  if (p == nullptr) return fail(KV4_EINVAL, "pool descriptor is NULL");
  if (p->fmt != KV4_NVFP4 && p->fmt != KV4_INT4_PTH && p->fmt != KV4_FP8 && p->fmt != KV4_K8V4)
    return fail(KV4_EINVAL, "bad fmt %d", p->fmt);
  if (p->reserved != 0) return fail(KV4_EINVAL, "pool.reserved must be 0");
  if (p->num_pages < 1) return fail(KV4_EINVAL, "num_pages must be >= 1");
  if (p->num_kv_heads < 1) return fail(KV4_EINVAL, "num_kv_heads must be >= 1");
  if (p->page_size < 16 || p->page_size % 16 != 0)
    return fail(KV4_EINVAL, "page_size %d is not a positive multiple of 16", p->page_size);
  if (p->head_dim != 64 && p->head_dim != 128 && p->head_dim != 256)
    return fail(KV4_EUNSUPPORTED, "head_dim %d not built (64, 128, 256)", p->head_dim);
  const int64_t bytes = static_cast<int64_t>(p->num_pages) * p->num_kv_heads * chunk_bytes_of(*p);
  if (bytes / (p->head_dim / 2) >= (int64_t{1} << 31))
    return fail(KV4_EUNSUPPORTED, "pool of %lld bytes exceeds the 2^31 code rows a TMA "
                "coordinate addresses", static_cast<long long>(bytes));
  return KV4_OK;
}

kv4_status check_pool_base(const kv4_pool* p) {
  if (p->base == nullptr) return fail(KV4_EINVAL, "pool.base is NULL");
  if (!aligned(p->base, 256)) return fail(KV4_EINVAL, "pool.base must be 256-byte aligned");
  return KV4_OK;
}

// ---------------------------------------------------------------- device state
__device__ int g_kv4_error_word;

int* error_word() {
  static int* cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (cache[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_kv4_error_word) != cudaSuccess) return nullptr;
    cache[dev] = static_cast<int*>(p);
  }
  return cache[dev];
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 152;
  return n;
}

// ---------------------------------------------------------------- TMA maps
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// The pool as a 2-D byte tensor of code rows: [pool_bytes / RB][RB], loaded in
// boxes of RB bytes x `box_rows` rows with the swizzle whose span is RB.
kv4_status code_row_map(const kv4_pool& p, int box_rows, CUtensorMap* map) {
  struct Entry { const void* base; int64_t rows; int rb; int box; CUtensorMap map; bool used; };
  static Entry cache[8];
  static int next = 0;
  static std::mutex mu;
  const int rb = p.head_dim / 2;
  const int64_t rows = static_cast<int64_t>(p.num_pages) * p.num_kv_heads * chunk_bytes_of(p) / rb;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (auto& e : cache)
      if (e.used && e.base == p.base && e.rows == rows && e.rb == rb && e.box == box_rows) {
        *map = e.map;
        return KV4_OK;
      }
  }
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return fail(KV4_ECUDA, "cuTensorMapEncodeTiled is not available");
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(rb), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(rb)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(rb), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle sw = rb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : rb == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                           : CU_TENSOR_MAP_SWIZZLE_32B;
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, p.base, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(KV4_ECUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  std::lock_guard<std::mutex> lock(mu);
  cache[next] = Entry{p.base, rows, rb, box_rows, *map, true};
  next = (next + 1) % 8;
  return KV4_OK;
}

// The two 3-D views the NVFP4 / INT4 decode kernel loads a 16-token tile
// through, each with one TMA copy per tile:
//  * codes: [2 (K, V: P code rows apart)][pool_bytes / RB rows][RB bytes],
//    box 16 rows x RB bytes x 2 (the tile's K rows, then its V rows), with the
//    swizzle whose span is RB;
//  * scales: [2 (K, V: P * SB bytes apart)][pool_bytes / (16 SB) rows][16 SB
//    bytes], box 1 row x 2 (the tile's 16 K scale rows, then its V rows).
// A chunk's scale region starts on a multiple of 16 SB bytes and a tile's
// first token is a multiple of 16, so every coordinate is whole.
kv4_status decode4_maps(const kv4_pool& p, CUtensorMap* codes, CUtensorMap* scales) {
  struct Entry { const void* base; int64_t bytes; int P, D, fmt; CUtensorMap c, s; bool used; };
  static Entry cache[8];
  static int next = 0;
  static std::mutex mu;
  const int64_t bytes = static_cast<int64_t>(p.num_pages) * p.num_kv_heads * chunk_bytes_of(p);
  {
    std::lock_guard<std::mutex> lock(mu);
    for (auto& e : cache)
      if (e.used && e.base == p.base && e.bytes == bytes && e.P == p.page_size && e.D == p.head_dim &&
          e.fmt == p.fmt) {
        *codes = e.c;
        *scales = e.s;
        return KV4_OK;
      }
  }
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return fail(KV4_ECUDA, "cuTensorMapEncodeTiled is not available");
  const int rb = p.head_dim / 2;
  auto swizzle_of = [](int row_bytes) {
    return row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
         : row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
  };
  if (p.fmt == KV4_K8V4) {
    // K: [chunk][token][line][KHB] (FP8 rows of D bytes as lines of at most 128);
    // V: [chunk][token][D/2] starting P*D bytes into each chunk.  The scales
    // are read with plain bulk copies.
    const int64_t nchunks = static_cast<int64_t>(p.num_pages) * p.num_kv_heads;
    const int khb = p.head_dim < 128 ? p.head_dim : 128, kh = p.head_dim / khb;
    const cuuint64_t cb = static_cast<cuuint64_t>(chunk_bytes_of(p));
    cuuint32_t e4[4] = {1, 1, 1, 1};
    {
      cuuint64_t dims[4] = {static_cast<cuuint64_t>(khb), static_cast<cuuint64_t>(kh),
                            static_cast<cuuint64_t>(p.page_size), static_cast<cuuint64_t>(nchunks)};
      cuuint64_t strides[3] = {static_cast<cuuint64_t>(khb), static_cast<cuuint64_t>(p.head_dim), cb};
      cuuint32_t box[4] = {static_cast<cuuint32_t>(khb), static_cast<cuuint32_t>(kh), 16, 1};
      CUresult r = fn(codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, p.base, dims, strides, box, e4,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_of(khb), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) return fail(KV4_ECUDA, "cuTensorMapEncodeTiled (k8v4 keys) failed (%d)", static_cast<int>(r));
    }
    {
      cuuint64_t dims[3] = {static_cast<cuuint64_t>(rb), static_cast<cuuint64_t>(p.page_size),
                            static_cast<cuuint64_t>(nchunks)};
      cuuint64_t strides[2] = {static_cast<cuuint64_t>(rb), cb};
      cuuint32_t box[3] = {static_cast<cuuint32_t>(rb), 16, 1};
      void* vbase = static_cast<uint8_t*>(p.base) + static_cast<int64_t>(p.page_size) * p.head_dim;
      CUresult r = fn(scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, vbase, dims, strides, box, e4,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_of(rb), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) return fail(KV4_ECUDA, "cuTensorMapEncodeTiled (k8v4 values) failed (%d)", static_cast<int>(r));
    }
    std::lock_guard<std::mutex> lock(mu);
    cache[next] = Entry{p.base, bytes, p.page_size, p.head_dim, p.fmt, *codes, *scales, true};
    next = (next + 1) % 8;
    return KV4_OK;
  }
  const int sb = p.fmt == KV4_NVFP4 ? p.head_dim / 16 : 4;
  const int srow = 16 * sb;
  if ((bytes / srow) >= (int64_t{1} << 31))
    return fail(KV4_EUNSUPPORTED, "pool of %lld bytes exceeds the 2^31 scale rows a TMA "
                "coordinate addresses", static_cast<long long>(bytes));
  const CUtensorMapSwizzle sw = rb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : rb == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                           : CU_TENSOR_MAP_SWIZZLE_32B;
  cuuint32_t estr[3] = {1, 1, 1};
  {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(rb), static_cast<cuuint64_t>(bytes / rb), 2};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(rb), static_cast<cuuint64_t>(p.page_size) * rb};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(rb), 16, 2};
    CUresult r = fn(codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, p.base, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(KV4_ECUDA, "cuTensorMapEncodeTiled (codes) failed (%d)", static_cast<int>(r));
  }
  {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(srow), static_cast<cuuint64_t>(bytes / srow), 2};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(srow), static_cast<cuuint64_t>(p.page_size) * sb};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(srow), 1, 2};
    CUresult r = fn(scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, p.base, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(KV4_ECUDA, "cuTensorMapEncodeTiled (scales) failed (%d)", static_cast<int>(r));
  }
  std::lock_guard<std::mutex> lock(mu);
  cache[next] = Entry{p.base, bytes, p.page_size, p.head_dim, p.fmt, *codes, *scales, true};
  next = (next + 1) % 8;
  return KV4_OK;
}

int64_t align256(int64_t x) { return (x + 255) / 256 * 256; }

}  // namespace

void kv4::set_error_message(const char* msg) { g_msg = msg; }

// Every argument check of kv4_decode_attention except the workspace's; shared
// with the static-workspace entry point so both report the same errors.
kv4_status kv4::check_decode_args(const void* q, const kv4_pool* pool,
                                  const float* layer_global_scale, const int32_t* block_table,
                                  int32_t max_pages, const int32_t* seq_lens, int32_t batch,
                                  int32_t num_q_heads, float sm_scale, int32_t num_splits,
                                  const void* out) {
  kv4_status s = check_pool(pool);
  if (s != KV4_OK) return s;
  if ((s = check_pool_base(pool)) != KV4_OK) return s;
  if (pool->fmt == KV4_K8V4)
    return fail(KV4_EUNSUPPORTED, "a k8v4 pool is read by kv4_k8v4_decode_attention");
  if (batch < 0) return fail(KV4_EINVAL, "batch < 0");
  if (num_q_heads < 1 || num_q_heads % pool->num_kv_heads != 0)
    return fail(KV4_EINVAL, "num_q_heads %d is not a positive multiple of num_kv_heads %d",
                num_q_heads, pool->num_kv_heads);
  if (max_pages < 1) return fail(KV4_EINVAL, "max_pages must be >= 1");
  if (static_cast<int64_t>(max_pages) * pool->page_size >= (int64_t{1} << 31))
    return fail(KV4_EINVAL, "max_pages * page_size must be < 2^31");
  if (num_splits < 0 || num_splits > 1024) return fail(KV4_EINVAL, "num_splits must be in [0, 1024]");
  if (!(sm_scale == sm_scale) || sm_scale > 3.0e38f || sm_scale < -3.0e38f)
    return fail(KV4_EINVAL, "sm_scale must be finite");
  if (batch == 0) return KV4_OK;
  if (q == nullptr || out == nullptr || block_table == nullptr || seq_lens == nullptr)
    return fail(KV4_EINVAL, "q, out, block_table and seq_lens must be non-NULL");
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(block_table, 4) || !aligned(seq_lens, 4))
    return fail(KV4_EINVAL, "q and out must be 16-byte aligned");
  if (pool->fmt != KV4_INT4_PTH && layer_global_scale == nullptr)
    return fail(KV4_EINVAL, "NVFP4 and FP8 need layer_global_scale");
  const int G = num_q_heads / pool->num_kv_heads;
  if (batch > 65535 || static_cast<int64_t>(pool->num_kv_heads) * ((G + 7) / 8) > 65535)
    return fail(KV4_EINVAL, "batch or heads exceed the launch grid");
  return KV4_OK;
}

extern "C" {

int64_t kv4_pool_chunk_bytes(const kv4_pool* pool) {
  if (check_pool(pool) != KV4_OK) return 0;
  return chunk_bytes_of(*pool);
}

int64_t kv4_pool_bytes(const kv4_pool* pool) {
  if (check_pool(pool) != KV4_OK) return 0;
  return static_cast<int64_t>(pool->num_pages) * pool->num_kv_heads * chunk_bytes_of(*pool);
}

static kv4_status write_common(const void* k, const void* v, const float* in_scale, bool fp8_in,
                               const int64_t* slot_mapping, int64_t num_tokens, const kv4_pool* pool,
                               const float* layer_global_scale, int32_t fmt, void* stream) {
  g_msg.clear();
  kv4_status s = check_pool(pool);
  if (s != KV4_OK) return s;
  if ((s = check_pool_base(pool)) != KV4_OK) return s;
  if (fmt != pool->fmt) return fail(KV4_EINVAL, "fmt %d does not match pool.fmt %d", fmt, pool->fmt);
  if (fmt == KV4_K8V4) return fail(KV4_EUNSUPPORTED, "a k8v4 pool is written by kv4_k8v4_write");
  if (num_tokens < 0) return fail(KV4_EINVAL, "num_tokens < 0");
  if (num_tokens == 0) return KV4_OK;
  if (k == nullptr || v == nullptr || slot_mapping == nullptr)
    return fail(KV4_EINVAL, "k, v and slot_mapping must be non-NULL");
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(slot_mapping, 8))
    return fail(KV4_EINVAL, "k and v must be 16-byte aligned, slot_mapping 8-byte aligned");
  if (fp8_in && (in_scale == nullptr || !aligned(in_scale, 4)))
    return fail(KV4_EINVAL, "the FP8 input needs its scales (in_scale, 4-byte aligned)");
  if (fmt != KV4_INT4_PTH && layer_global_scale == nullptr)
    return fail(KV4_EINVAL, "NVFP4 and FP8 need layer_global_scale");
  const int64_t threads = num_tokens * pool->num_kv_heads * (pool->head_dim / 8);
  if (threads >= (int64_t{1} << 31))           // thread indices are 32-bit
    return fail(KV4_EINVAL, "num_tokens too large");

  kv4::WriteArgs a{};
  if (fp8_in) {
    a.k8 = static_cast<const uint8_t*>(k);
    a.v8 = static_cast<const uint8_t*>(v);
    a.in_scale = in_scale;
  } else {
    a.k = static_cast<const __nv_bfloat16*>(k);
    a.v = static_cast<const __nv_bfloat16*>(v);
  }
  a.slot_mapping = slot_mapping;
  a.T = num_tokens;
  a.pool = static_cast<uint8_t*>(pool->base);
  a.chunk_bytes = chunk_bytes_of(*pool);
  a.P = pool->page_size;
  a.Hkv = pool->num_kv_heads;
  a.num_pages = pool->num_pages;
  a.D = pool->head_dim;
  a.fmt = fmt;
  a.gscale = layer_global_scale;
  a.sms = sm_count();
  a.err = error_word();
  if (a.err == nullptr) return fail(KV4_ECUDA, "no CUDA device / error word unavailable");
  cudaError_t e = kv4::launch_write(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KV4_OK : cuda_fail(e, fp8_in ? "kv4_write_fp8 launch" : "kv4_write launch");
}

kv4_status kv4_write(const void* k, const void* v, const int64_t* slot_mapping,
                     int64_t num_tokens, const kv4_pool* pool,
                     const float* layer_global_scale, int32_t fmt, void* stream) {
  kv4::NvtxRange nvtx_range("kv4_write");
  return write_common(k, v, nullptr, false, slot_mapping, num_tokens, pool, layer_global_scale, fmt,
                      stream);
}

kv4_status kv4_write_fp8(const void* k, const void* v, const float* in_scale,
                         const int64_t* slot_mapping, int64_t num_tokens, const kv4_pool* pool,
                         const float* layer_global_scale, int32_t fmt, void* stream) {
  kv4::NvtxRange nvtx_range("kv4_write_fp8");
  return write_common(k, v, in_scale, true, slot_mapping, num_tokens, pool, layer_global_scale, fmt,
                      stream);
}

int64_t kv4_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t head_dim,
                                   int32_t num_splits) {
  if (batch < 0 || num_q_heads < 0 || head_dim < 0 || num_splits < 0) return 0;
  if (num_splits == 1 || batch == 0) return 0;        // one CTA per unit writes `out` directly
  const int64_t S = num_splits == 0 ? 1 : num_splits;
  // units (request, kv head, slice of <= 8 query heads) number at most batch * num_q_heads
  const int64_t slots = static_cast<int64_t>(sm_count()) * kv4::decode_max_ctas_per_sm() +
                        static_cast<int64_t>(batch) * num_q_heads * S;
  return align256((batch + 1) * 8) + align256(slots * 8 * 16) + slots * 8 * head_dim * 4;
}

// kv4_decode_attention, and kv4_decode_step when k_new / v_new are given.
static kv4_status decode_common(const void* q, const void* k_new, const void* v_new, const kv4_pool* pool,
                                const float* layer_global_scale, const int32_t* block_table,
                                int32_t max_pages, const int32_t* seq_lens, int32_t batch,
                                int32_t num_q_heads, float sm_scale, int32_t num_splits,
                                void* workspace, int64_t workspace_bytes, void* out,
                                int32_t out_is_fp32, void* stream) {
  g_msg.clear();
  kv4_status s = kv4::check_decode_args(q, pool, layer_global_scale, block_table, max_pages,
                                        seq_lens, batch, num_q_heads, sm_scale, num_splits, out);
  if (s != KV4_OK || batch == 0) return s;
  if (k_new != nullptr || v_new != nullptr) {
    if (pool->fmt != KV4_NVFP4 && pool->fmt != KV4_INT4_PTH)
      return fail(KV4_EUNSUPPORTED, "kv4_decode_step: NVFP4 and INT4 pools only (use kv4_write, then decode)");
    if (num_q_heads / pool->num_kv_heads > 8)
      return fail(KV4_EUNSUPPORTED, "kv4_decode_step: at most 8 query heads per kv head");
    if (k_new == nullptr || v_new == nullptr) return fail(KV4_EINVAL, "k_new and v_new must be non-NULL");
    if (!aligned(k_new, 16) || !aligned(v_new, 16)) return fail(KV4_EINVAL, "k_new and v_new must be 16-byte aligned");
  }
  const int G = num_q_heads / pool->num_kv_heads;
  const int64_t need = kv4_decode_workspace_bytes(batch, num_q_heads, pool->head_dim, num_splits);
  if (need > 0) {
    if (workspace == nullptr || workspace_bytes < need)
      return fail(KV4_EINVAL, "workspace of %lld bytes needed for num_splits %d",
                  static_cast<long long>(need), num_splits);
    if (!aligned(workspace, 256)) return fail(KV4_EINVAL, "workspace must be 256-byte aligned");
  }
  const int64_t units = static_cast<int64_t>(batch) * pool->num_kv_heads * ((G + 7) / 8);
  if (units >= (int64_t{1} << 31)) return fail(KV4_EINVAL, "too many (request, head) units");

  kv4::DecodeArgs a{};
  a.pool = static_cast<const uint8_t*>(pool->base);
  a.chunk_bytes = chunk_bytes_of(*pool);
  a.P = pool->page_size;
  a.Hkv = pool->num_kv_heads;
  a.num_pages = pool->num_pages;
  a.D = pool->head_dim;
  a.fmt = pool->fmt;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.gscale = layer_global_scale;
  a.block_table = block_table;
  a.max_pages = max_pages;
  a.seq_lens = seq_lens;
  a.B = batch;
  a.Hq = num_q_heads;
  a.G = G;
  a.sm_scale = sm_scale;
  if (num_splits == 1) {
    a.num_splits = 1;
    a.unit_ctas = 1;
    a.n_cta = static_cast<int>(units);
  } else {
    // one wave of persistent CTAs, each given an equal share of all tiles
    const int64_t tiles_max = units * ((static_cast<int64_t>(max_pages) * pool->page_size +
                                        kv4::decode_tile_tokens(pool->fmt) - 1) /
                                       kv4::decode_tile_tokens(pool->fmt));
    const int64_t resident = static_cast<int64_t>(sm_count()) * kv4::decode_ctas_per_sm(pool->fmt);
    // at least a few tiles per compute warp
    const int64_t min_tiles = pool->fmt == KV4_FP8 ? 4 : 12;
    int64_t n = (tiles_max + min_tiles - 1) / min_tiles;
    n = n < 1 ? 1 : (n > resident ? resident : n);
    a.num_splits = num_splits == 0 ? 1 : num_splits;
    a.unit_ctas = 0;
    a.n_cta = static_cast<int>(n);
    const int64_t slots = static_cast<int64_t>(sm_count()) * kv4::decode_max_ctas_per_sm() +
                          static_cast<int64_t>(batch) * num_q_heads * a.num_splits;
    uint8_t* w = static_cast<uint8_t*>(workspace);
    a.cum = reinterpret_cast<int64_t*>(w);
    a.part_ml = reinterpret_cast<float*>(w + align256((batch + 1) * 8));
    a.part_o = reinterpret_cast<float*>(w + align256((batch + 1) * 8) + align256(slots * 8 * 16));
  }
  a.out = out;
  a.out_f32 = out_is_fp32 ? 1 : 0;
  a.err = error_word();
  if (a.err == nullptr) return fail(KV4_ECUDA, "no CUDA device / error word unavailable");
  a.tile = kv4::decode_tile_tokens(pool->fmt);
  // a tile is 16 tokens: one box of 16 code rows (NVFP4, INT4) or 32 (FP8,
  // two code rows a token)
  a.box_rows = pool->fmt == KV4_FP8 ? 32 : 16;
  CUtensorMap map, map2;
  if (pool->fmt == KV4_FP8) {
    if ((s = code_row_map(*pool, a.box_rows, &map)) != KV4_OK) return s;
    map2 = map;
  } else if ((s = decode4_maps(*pool, &map, &map2)) != KV4_OK) {
    return s;
  }
  a.k_new = static_cast<const __nv_bfloat16*>(k_new);
  a.v_new = static_cast<const __nv_bfloat16*>(v_new);
  cudaError_t e = kv4::launch_decode(a, map, map2, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KV4_OK : cuda_fail(e, "kv4_decode_attention launch");
}

kv4_status kv4_decode_attention(const void* q, const kv4_pool* pool,
                                const float* layer_global_scale, const int32_t* block_table,
                                int32_t max_pages, const int32_t* seq_lens, int32_t batch,
                                int32_t num_q_heads, float sm_scale, int32_t num_splits,
                                void* workspace, int64_t workspace_bytes, void* out,
                                int32_t out_is_fp32, void* stream) {
  kv4::NvtxRange nvtx_range("kv4_decode_attention");
  return decode_common(q, nullptr, nullptr, pool, layer_global_scale, block_table, max_pages, seq_lens, batch,
                       num_q_heads, sm_scale, num_splits, workspace, workspace_bytes, out, out_is_fp32, stream);
}

kv4_status kv4_decode_step(const void* q, const void* k_new, const void* v_new, const kv4_pool* pool,
                           const float* layer_global_scale, const int32_t* block_table,
                           int32_t max_pages, const int32_t* seq_lens, int32_t batch,
                           int32_t num_q_heads, float sm_scale, int32_t num_splits,
                           void* workspace, int64_t workspace_bytes, void* out,
                           int32_t out_is_fp32, void* stream) {
  kv4::NvtxRange nvtx_range("kv4_decode_step");
  if (k_new == nullptr || v_new == nullptr) {
    g_msg.clear();
    return fail(KV4_EINVAL, "kv4_decode_step: k_new and v_new must be non-NULL");
  }
  return decode_common(q, k_new, v_new, pool, layer_global_scale, block_table, max_pages, seq_lens, batch,
                       num_q_heads, sm_scale, num_splits, workspace, workspace_bytes, out, out_is_fp32, stream);
}

kv4_status kv4_calibrate_global_scale(const void* k, const void* v, int64_t num_tokens,
                                      int32_t num_kv_heads, int32_t head_dim,
                                      float* layer_global_scale, void* stream) {
  kv4::NvtxRange nvtx_range("kv4_calibrate_global_scale");
  g_msg.clear();
  if (num_tokens < 0 || num_kv_heads < 1) return fail(KV4_EINVAL, "num_tokens < 0 or num_kv_heads < 1");
  if (head_dim != 64 && head_dim != 128 && head_dim != 256)
    return fail(KV4_EUNSUPPORTED, "head_dim %d not built (64, 128, 256)", head_dim);
  if (layer_global_scale == nullptr || !aligned(layer_global_scale, 8))
    return fail(KV4_EINVAL, "layer_global_scale must be a non-NULL, 8-byte aligned float[2]");
  if (num_tokens > 0 && (k == nullptr || v == nullptr || !aligned(k, 16) || !aligned(v, 16)))
    return fail(KV4_EINVAL, "k and v must be non-NULL and 16-byte aligned");
  kv4::CalibArgs a{};
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.v = static_cast<const __nv_bfloat16*>(v);
  a.n = num_tokens * num_kv_heads * head_dim;
  a.out = layer_global_scale;
  cudaError_t e = kv4::launch_calibrate(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KV4_OK : cuda_fail(e, "kv4_calibrate_global_scale launch");
}

kv4_status kv4_dequant_prefix(const kv4_pool* pool, const float* layer_global_scale,
                              const int32_t* block_table, int32_t max_pages,
                              const int32_t* prefix_lens, const int64_t* cu_prefix,
                              int32_t batch, int32_t max_prefix_len, const float* fp8_scale,
                              void* fp8_k, void* fp8_v, void* stream) {
  kv4::NvtxRange nvtx_range("kv4_dequant_prefix");
  g_msg.clear();
  kv4_status s = check_pool(pool);
  if (s != KV4_OK) return s;
  if ((s = check_pool_base(pool)) != KV4_OK) return s;
  if (pool->fmt == KV4_FP8)
    return fail(KV4_EUNSUPPORTED, "an FP8 pool is already FP8: no prefix dequant");
  if (pool->fmt == KV4_K8V4)
    return fail(KV4_EUNSUPPORTED, "no prefix dequant for a k8v4 pool");
  if (batch < 0 || max_prefix_len < 0) return fail(KV4_EINVAL, "batch and max_prefix_len must be >= 0");
  if (max_pages < 1) return fail(KV4_EINVAL, "max_pages must be >= 1");
  if (static_cast<int64_t>(max_pages) * pool->page_size >= (int64_t{1} << 31))
    return fail(KV4_EINVAL, "max_pages * page_size must be < 2^31");
  if (max_prefix_len > max_pages * pool->page_size)
    return fail(KV4_EINVAL, "max_prefix_len exceeds max_pages * page_size");
  if (batch > 65535) return fail(KV4_EINVAL, "batch exceeds the launch grid");
  if (batch == 0 || max_prefix_len == 0) return KV4_OK;
  if (block_table == nullptr || prefix_lens == nullptr || cu_prefix == nullptr ||
      fp8_scale == nullptr || fp8_k == nullptr || fp8_v == nullptr)
    return fail(KV4_EINVAL, "block_table, prefix_lens, cu_prefix, fp8_scale and outputs must be non-NULL");
  if (!aligned(fp8_k, 16) || !aligned(fp8_v, 16) || !aligned(cu_prefix, 8) || !aligned(fp8_scale, 4) ||
      !aligned(block_table, 4) || !aligned(prefix_lens, 4) ||
      (layer_global_scale != nullptr && !aligned(layer_global_scale, 4)))
    return fail(KV4_EINVAL, "fp8_k and fp8_v must be 16-byte aligned (int64 arrays 8-byte, others 4-byte)");
  if (pool->fmt == KV4_NVFP4 && layer_global_scale == nullptr)
    return fail(KV4_EINVAL, "NVFP4 needs layer_global_scale");
  const int64_t threads = static_cast<int64_t>(max_prefix_len) * pool->num_kv_heads * (pool->head_dim / 16);
  if (threads >= (int64_t{1} << 31)) return fail(KV4_EINVAL, "prefix too large");  // 32-bit thread indices

  kv4::PrefixArgs a{};
  a.pool = static_cast<const uint8_t*>(pool->base);
  a.chunk_bytes = chunk_bytes_of(*pool);
  a.P = pool->page_size;
  a.Hkv = pool->num_kv_heads;
  a.num_pages = pool->num_pages;
  a.D = pool->head_dim;
  a.fmt = pool->fmt;
  a.gscale = layer_global_scale;
  a.block_table = block_table;
  a.max_pages = max_pages;
  a.prefix_lens = prefix_lens;
  a.cu_prefix = cu_prefix;
  a.B = batch;
  a.max_prefix_len = max_prefix_len;
  a.fp8_scale = fp8_scale;
  a.out_k = static_cast<uint8_t*>(fp8_k);
  a.out_v = static_cast<uint8_t*>(fp8_v);
  a.err = error_word();
  if (a.err == nullptr) return fail(KV4_ECUDA, "no CUDA device / error word unavailable");
  a.sms = sm_count();
  // the workspaces as 2-D byte tensors of 128-byte rows for the kernel's
  // tensor stores; the extent is not the buffers' (the offsets come from the
  // device array cu_prefix): the kernel stores only the rows of its items
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return fail(KV4_ECUDA, "cuTensorMapEncodeTiled is not available");
  CUtensorMap maps[2];
  for (int i = 0; i < 2; ++i) {
    cuuint64_t dims[2] = {128, cuuint64_t{1} << 31};
    cuuint64_t strides[1] = {128};
    cuuint32_t box[2] = {128, 16};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(&maps[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, i == 0 ? fp8_k : fp8_v, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
      return fail(KV4_ECUDA, "cuTensorMapEncodeTiled (prefix workspace) failed (%d)", static_cast<int>(r));
  }
  cudaError_t e = kv4::launch_prefix(a, maps[0], maps[1], static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KV4_OK : cuda_fail(e, "kv4_dequant_prefix launch");
}

int64_t kv4_extend_workspace_bytes(int32_t batch, int32_t max_chunk_len, int32_t num_q_heads,
                                   int32_t head_dim) {
  if (batch <= 0 || max_chunk_len <= 0 || num_q_heads <= 0 || head_dim <= 0) return 0;
  const int64_t items = static_cast<int64_t>(batch) * ((static_cast<int64_t>(max_chunk_len) + 127) / 128) * num_q_heads;
  if (items >= (int64_t{1} << 31)) return 0;
  int split = 0, ways = 1;
  kv4::extend_split(static_cast<int>(items), sm_count(), split, ways);
  const int64_t pieces = static_cast<int64_t>(split) * ways;
  return align256(pieces * 128 * head_dim * 4) + pieces * 128 * 8;
}

kv4_status kv4_extend_attention(const void* q, const void* chunk_k, const void* chunk_v,
                                const void* prefix_k, const void* prefix_v,
                                const float* fp8_scale, const int32_t* prefix_lens,
                                const int64_t* cu_prefix, const int32_t* chunk_lens,
                                const int64_t* cu_chunk, int32_t batch, int32_t max_chunk_len,
                                int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                float sm_scale, void* workspace, int64_t workspace_bytes, void* out,
                                int32_t out_is_fp32, void* stream) {
  kv4::NvtxRange nvtx_range("kv4_extend_attention");
  g_msg.clear();
  if (batch < 0 || max_chunk_len < 0) return fail(KV4_EINVAL, "batch and max_chunk_len must be >= 0");
  if (num_kv_heads < 1 || num_q_heads < 1 || num_q_heads % num_kv_heads != 0)
    return fail(KV4_EINVAL, "num_q_heads must be a positive multiple of num_kv_heads");
  if (head_dim != 64 && head_dim != 128 && head_dim != 256)
    return fail(KV4_EUNSUPPORTED, "head_dim %d not built (64, 128, 256)", head_dim);
  if (!(sm_scale > 0.f) || !(sm_scale < 3.0e38f)) return fail(KV4_EINVAL, "sm_scale must be positive and finite");
  if (batch > 65535) return fail(KV4_EINVAL, "batch exceeds the launch grid");
  if ((static_cast<int64_t>(max_chunk_len) + 127) / 128 > 65535)
    return fail(KV4_EINVAL, "max_chunk_len exceeds the launch grid");
  if (batch == 0 || max_chunk_len == 0) return KV4_OK;
  const int64_t items = static_cast<int64_t>(batch) * ((static_cast<int64_t>(max_chunk_len) + 127) / 128) * num_q_heads;
  if (items >= (int64_t{1} << 31)) return fail(KV4_EINVAL, "too many (request, query tile, head) items");
  if (q == nullptr || chunk_k == nullptr || chunk_v == nullptr || prefix_k == nullptr ||
      prefix_v == nullptr || fp8_scale == nullptr || prefix_lens == nullptr ||
      cu_prefix == nullptr || chunk_lens == nullptr || cu_chunk == nullptr || out == nullptr)
    return fail(KV4_EINVAL, "device pointers must be non-NULL");
  if (!aligned(q, 16) || !aligned(chunk_k, 16) || !aligned(chunk_v, 16) || !aligned(prefix_k, 16) ||
      !aligned(prefix_v, 16) || !aligned(out, 16) || !aligned(cu_prefix, 8) || !aligned(cu_chunk, 8) ||
      !aligned(fp8_scale, 4) || !aligned(prefix_lens, 4) || !aligned(chunk_lens, 4))
    return fail(KV4_EINVAL, "device buffers must be 16-byte aligned (int64 arrays 8-byte)");

  kv4::ExtendArgs a{};
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.ck = static_cast<const uint8_t*>(chunk_k);
  a.cv = static_cast<const uint8_t*>(chunk_v);
  a.pk = static_cast<const uint8_t*>(prefix_k);
  a.pv = static_cast<const uint8_t*>(prefix_v);
  a.fp8_scale = fp8_scale;
  a.prefix_lens = prefix_lens;
  a.cu_prefix = cu_prefix;
  a.chunk_lens = chunk_lens;
  a.cu_chunk = cu_chunk;
  a.B = batch;
  a.max_chunk_len = max_chunk_len;
  a.Hq = num_q_heads;
  a.Hkv = num_kv_heads;
  a.D = head_dim;
  a.G = num_q_heads / num_kv_heads;
  a.sm_scale = sm_scale;
  a.out = out;
  a.out_f32 = out_is_fp32 ? 1 : 0;
  a.qtiles = (max_chunk_len + 127) / 128;
  a.items = static_cast<int>(items);
  a.split = 0;
  a.ways = 1;
  if (workspace != nullptr) {
    // the remainder of the last wave split into key-range pieces
    const int64_t need = kv4_extend_workspace_bytes(batch, max_chunk_len, num_q_heads, head_dim);
    if (workspace_bytes < need)
      return fail(KV4_EINVAL, "workspace of %lld bytes is smaller than the %lld needed",
                  static_cast<long long>(workspace_bytes), static_cast<long long>(need));
    if (!aligned(workspace, 256)) return fail(KV4_EINVAL, "workspace must be 256-byte aligned");
    kv4::extend_split(a.items, sm_count(), a.split, a.ways);
    const int64_t pieces = static_cast<int64_t>(a.split) * a.ways;
    a.part_o = static_cast<float*>(workspace);
    a.part_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + align256(pieces * 128 * head_dim * 4));
  }
  a.err = error_word();
  if (a.err == nullptr) return fail(KV4_ECUDA, "no CUDA device / error word unavailable");
  cudaError_t e = kv4::launch_extend(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KV4_OK : cuda_fail(e, "kv4_extend_attention launch");
}

kv4_status kv4_k8v4_write(const void* k, const void* v, const int64_t* slot_mapping,
                          int64_t num_tokens, const kv4_pool* pool, const float* key_scale,
                          void* stream) {
  kv4::NvtxRange nvtx_range("kv4_k8v4_write");
  g_msg.clear();
  kv4_status s = check_pool(pool);
  if (s != KV4_OK) return s;
  if ((s = check_pool_base(pool)) != KV4_OK) return s;
  if (pool->fmt != KV4_K8V4) return fail(KV4_EINVAL, "pool.fmt must be KV4_K8V4");
  if (num_tokens < 0) return fail(KV4_EINVAL, "num_tokens < 0");
  if (num_tokens == 0) return KV4_OK;
  if (k == nullptr || v == nullptr || slot_mapping == nullptr || key_scale == nullptr)
    return fail(KV4_EINVAL, "k, v, slot_mapping and key_scale must be non-NULL");
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(slot_mapping, 8) || !aligned(key_scale, 4))
    return fail(KV4_EINVAL, "k and v must be 16-byte aligned, slot_mapping 8-byte aligned");
  if (num_tokens * pool->num_kv_heads >= (int64_t{1} << 31))   // 32-bit row indices
    return fail(KV4_EINVAL, "num_tokens too large");
  kv4::K8V4WriteArgs a{};
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.v = static_cast<const __nv_bfloat16*>(v);
  a.slot_mapping = slot_mapping;
  a.rows = num_tokens * pool->num_kv_heads;
  a.pool = static_cast<uint8_t*>(pool->base);
  a.chunk_bytes = chunk_bytes_of(*pool);
  a.P = pool->page_size;
  a.Hkv = pool->num_kv_heads;
  a.num_pages = pool->num_pages;
  a.D = pool->head_dim;
  a.s_k = key_scale;
  a.err = error_word();
  if (a.err == nullptr) return fail(KV4_ECUDA, "no CUDA device / error word unavailable");
  cudaError_t e = kv4::launch_k8v4_write(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KV4_OK : cuda_fail(e, "kv4_k8v4_write launch");
}

int64_t kv4_k8v4_workspace_bytes(int32_t batch, int32_t num_kv_heads, int32_t head_dim,
                                 int32_t num_chunks) {
  if (batch < 0 || num_kv_heads < 0 || head_dim < 0 || num_chunks < 1) return 0;
  // the layout of kv4_decode_attention's: tile offsets, piece states, piece
  // outputs; a unit is one (request, kv head) with its <= 8 query heads
  const int64_t slots = static_cast<int64_t>(sm_count()) * kv4::decode_max_ctas_per_sm() +
                        static_cast<int64_t>(batch) * num_kv_heads * num_chunks;
  return align256((static_cast<int64_t>(batch) + 1) * 8) + align256(slots * 8 * 16) + slots * 8 * head_dim * 4;
}

kv4_status kv4_k8v4_decode_attention(const void* q, const kv4_pool* pool, const float* key_scale,
                                     const int32_t* block_table, int32_t max_pages,
                                     const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                                     float sm_scale, int32_t num_chunks, void* workspace,
                                     int64_t workspace_bytes, void* out, int32_t out_is_fp32,
                                     void* stream) {
  kv4::NvtxRange nvtx_range("kv4_k8v4_decode_attention");
  g_msg.clear();
  kv4_status s = check_pool(pool);
  if (s != KV4_OK) return s;
  if ((s = check_pool_base(pool)) != KV4_OK) return s;
  if (pool->fmt != KV4_K8V4) return fail(KV4_EINVAL, "pool.fmt must be KV4_K8V4");
  if (batch < 0 || batch > 65535) return fail(KV4_EINVAL, "batch must be in [0, 65535]");
  if (num_q_heads < 1 || num_q_heads % pool->num_kv_heads != 0)
    return fail(KV4_EINVAL, "num_q_heads must be a positive multiple of num_kv_heads");
  if (num_q_heads / pool->num_kv_heads > 8)
    return fail(KV4_EUNSUPPORTED, "k8v4 decode supports at most 8 query heads per kv head");
  if (num_chunks < 1 || num_chunks > 65535) return fail(KV4_EINVAL, "num_chunks must be in [1, 65535]");
  if (max_pages < 1) return fail(KV4_EINVAL, "max_pages must be >= 1");
  if (static_cast<int64_t>(max_pages) * pool->page_size >= (int64_t{1} << 31))
    return fail(KV4_EINVAL, "max_pages * page_size must be < 2^31");
  if (!(sm_scale > 0.f) || !(sm_scale < 3.0e38f)) return fail(KV4_EINVAL, "sm_scale must be positive and finite");
  if (batch == 0) return KV4_OK;
  if (q == nullptr || key_scale == nullptr || block_table == nullptr || seq_lens == nullptr ||
      out == nullptr || workspace == nullptr)
    return fail(KV4_EINVAL, "q, key_scale, block_table, seq_lens, workspace and out must be non-NULL");
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(workspace, 256) || !aligned(key_scale, 4) ||
      !aligned(block_table, 4) || !aligned(seq_lens, 4))
    return fail(KV4_EINVAL, "q and out must be 16-byte aligned, workspace 256-byte aligned");
  const int64_t need = kv4_k8v4_workspace_bytes(batch, pool->num_kv_heads, pool->head_dim, num_chunks);
  if (workspace_bytes < need)
    return fail(KV4_EINVAL, "workspace of %lld bytes is smaller than the %lld needed",
                static_cast<long long>(workspace_bytes), static_cast<long long>(need));
  const int64_t units = static_cast<int64_t>(batch) * pool->num_kv_heads;

  // the NVFP4 / INT4 decode kernel with FP8 keys and rotated queries, always
  // through the combine (which rotates the output back)
  kv4::DecodeArgs a{};
  a.pool = static_cast<const uint8_t*>(pool->base);
  a.chunk_bytes = chunk_bytes_of(*pool);
  a.P = pool->page_size;
  a.Hkv = pool->num_kv_heads;
  a.num_pages = pool->num_pages;
  a.D = pool->head_dim;
  a.fmt = KV4_K8V4;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.gscale = key_scale;
  a.block_table = block_table;
  a.max_pages = max_pages;
  a.seq_lens = seq_lens;
  a.B = batch;
  a.Hq = num_q_heads;
  a.G = num_q_heads / pool->num_kv_heads;
  a.sm_scale = sm_scale;
  a.tile = kv4::decode_tile_tokens(KV4_K8V4);
  const int64_t tiles_max = units * ((static_cast<int64_t>(max_pages) * pool->page_size + a.tile - 1) / a.tile);
  const int64_t resident = static_cast<int64_t>(sm_count()) * kv4::decode_ctas_per_sm(KV4_K8V4);
  int64_t n = (tiles_max + 11) / 12;       // at least a few tiles per compute warp
  n = n < 1 ? 1 : (n > resident ? resident : n);
  a.num_splits = num_chunks;
  a.unit_ctas = 0;
  a.n_cta = static_cast<int>(n);
  const int64_t slots = static_cast<int64_t>(sm_count()) * kv4::decode_max_ctas_per_sm() + units * num_chunks;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  a.cum = reinterpret_cast<int64_t*>(w);
  a.part_ml = reinterpret_cast<float*>(w + align256((static_cast<int64_t>(batch) + 1) * 8));
  a.part_o = reinterpret_cast<float*>(w + align256((static_cast<int64_t>(batch) + 1) * 8) + align256(slots * 8 * 16));
  a.out = out;
  a.out_f32 = out_is_fp32 ? 1 : 0;
  a.err = error_word();
  if (a.err == nullptr) return fail(KV4_ECUDA, "no CUDA device / error word unavailable");
  CUtensorMap kmap, vmap;
  if ((s = decode4_maps(*pool, &kmap, &vmap)) != KV4_OK) return s;
  cudaError_t e = kv4::launch_decode(a, kmap, vmap, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KV4_OK : cuda_fail(e, "kv4_k8v4_decode_attention launch");
}

int32_t kv4_device_error(void) {
  int* p = error_word();
  if (p == nullptr) return KV4_ECUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return KV4_ECUDA;
  int v = 0;
  if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return KV4_ECUDA;
  const int zero = 0;
  if (cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return KV4_ECUDA;
  return v;
}

const char* kv4_status_str(int32_t status) {
  switch (status) {
    case KV4_OK: return "KV4_OK";
    case KV4_EINVAL: return "KV4_EINVAL: invalid argument";
    case KV4_EUNSUPPORTED: return "KV4_EUNSUPPORTED: shape not supported";
    case KV4_ECUDA: return "KV4_ECUDA: CUDA runtime error";
    case KV4_EBOUNDS: return "KV4_EBOUNDS: index outside the pool or table";
    case KV4_ETIMEOUT: return "KV4_ETIMEOUT: a bounded wait ran out";
    default: return "KV4: unknown status";
  }
}

const char* kv4_last_error_message(void) { return g_msg.c_str(); }

}  // extern "C"
