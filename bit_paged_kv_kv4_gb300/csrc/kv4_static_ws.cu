// kv4_decode_attention_static_ws: decode attention whose split scratch lives
// in a fixed device array owned by the library, for callers that cannot
// allocate device memory themselves.
//
// Who needs it: code that runs inside a host framework which owns every device
// allocation (an inference-server plugin with a fixed memory budget, say), or a
// decode loop that cannot afford the device-wide synchronisation cudaMalloc /
// cudaFree may trigger.  Such a caller passes its inputs and outputs as usual;
// the per-split partial results go to kScratch below instead of a
// caller-provided workspace.
//
// Rules of the shared array:
//  * It is kKv4StaticWorkspaceBytes (8 MiB) and exists on every GPU that loads
//    the library, for the life of the process.
//  * Host code cannot pass `kScratch` itself to a kernel (on the host it names
//    a stand-in, not the device copy), so the first call on each device looks up
//    the device address with cudaGetSymbolAddress while that device is current
//    and caches it.  Make that first call before any stream capture.  The
//    cached address belongs to the device's context of that moment:
//    cudaDeviceReset discards it with the rest of the library's device state,
//    so a process that resets a device must not call here on it again.
//  * Every call shares the one array and it keeps the last call's contents.
//    Nothing in it has to start at zero: each call writes every partial before
//    the combine step reads it.  Calls whose kernels overlap on the GPU (two
//    streams, or two host threads) race on the array and give wrong results.
//  * A call whose batch x query heads x splits needs more than the array holds
//    is rejected with KV4_EINVAL and a message giving both sizes.
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "../../include/kv4.h"
#include "kv4_internal.h"

namespace {

constexpr int64_t kKv4StaticWorkspaceBytes = int64_t{8} << 20;

static __device__ __align__(256) unsigned char kScratch[kKv4StaticWorkspaceBytes];

// Device address of kScratch on the current device, looked up once per device.
kv4_status scratch_address(void** out) {
  static void* addr[64] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    kv4::set_error_message("kv4_decode_attention_static_ws: no usable CUDA device");
    return KV4_ECUDA;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, kScratch);
    if (e != cudaSuccess || p == nullptr) {
      char buf[256];
      snprintf(buf, sizeof(buf),
               "kv4_decode_attention_static_ws: cudaGetSymbolAddress failed on device %d: %s",
               dev, cudaGetErrorString(e));
      kv4::set_error_message(buf);
      return KV4_ECUDA;
    }
    addr[dev] = p;
  }
  *out = addr[dev];
  return KV4_OK;
}

}  // namespace

extern "C" {

kv4_status kv4_decode_attention_static_ws(const void* q, const kv4_pool* pool,
                                          const float* layer_global_scale,
                                          const int32_t* block_table, int32_t max_pages,
                                          const int32_t* seq_lens, int32_t batch,
                                          int32_t num_q_heads, float sm_scale,
                                          int32_t num_splits, void* out, int32_t out_is_fp32,
                                          void* stream) {
  kv4::NvtxRange nvtx_range("kv4_decode_attention_static_ws");
  // the argument checks of kv4_decode_attention come first, so an invalid call
  // gets the same precise message as there, not the scratch-size one below
  kv4::set_error_message("");
  kv4_status s = kv4::check_decode_args(q, pool, layer_global_scale, block_table, max_pages,
                                        seq_lens, batch, num_q_heads, sm_scale, num_splits, out);
  if (s != KV4_OK || batch == 0) return s;
  const int64_t need = kv4_decode_workspace_bytes(batch, num_q_heads, pool->head_dim, num_splits);
  if (need > kKv4StaticWorkspaceBytes) {
    char buf[256];
    snprintf(buf, sizeof(buf),
             "kv4_decode_attention_static_ws: %d requests x %d query heads with num_splits %d "
             "need %lld bytes of scratch; the static workspace holds %lld",
             batch, num_q_heads, num_splits, static_cast<long long>(need),
             static_cast<long long>(kKv4StaticWorkspaceBytes));
    kv4::set_error_message(buf);
    return KV4_EINVAL;
  }
  void* ws = nullptr;
  if (need > 0) {
    s = scratch_address(&ws);
    if (s != KV4_OK) return s;
  }
  return kv4_decode_attention(q, pool, layer_global_scale, block_table, max_pages, seq_lens,
                              batch, num_q_heads, sm_scale, num_splits, ws, need > 0 ? need : 0, out,
                              out_is_fp32, stream);
}

}  // extern "C"
