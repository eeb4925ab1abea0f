// Serving-time calibration of the NVFP4 global scales ("SGLang's 4-bit KV
// cache", Figure 2: per-layer FP32 global scales; the caveat above "The
// agentic result": the measured runs went without them, and calibrating them
// is named as unfinished work).  g = float32(amax) / 2688 (E2M1 max x E4M3 max), one
// FP32 rounding, and g = 1 when amax is not positive.
//
// amax_kernel: every thread takes 8 bf16 per 16-byte load, four loads in
// flight, in a grid-stride loop, and keeps the largest |x| as bits (a
// non-negative float's bit pattern orders like the float); warps and the
// block reduce it and one atomicMax per block lands in the caller's output
// word, which zero_kernel cleared first.  finalize_kernel turns the two
// maxima into the scales.  The three are chained by programmatic dependent
// launch, so the reductions stream while the zeroing drains.
// The maximum is exact and order-free, so the result is deterministic.
#include <cstdint>

#include "kv4_device.cuh"
#include "kv4_internal.h"

namespace kv4 {

__global__ void __launch_bounds__(256)
amax_kernel(const CalibArgs a) {
  grid_dep_launch();   // finalize_kernel may be scheduled; it waits for this grid
  // The inputs are read before grid_dep_wait(): the kernel before this one is
  // zero_kernel, an ordinary launch, so whatever produced them had completed
  // when it started.
  const uint4* src = reinterpret_cast<const uint4*>(blockIdx.y == 0 ? a.k : a.v);
  const int64_t n8 = a.n / 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  uint32_t m = 0;
  auto fold = [&m](const uint4 w) {
    const uint32_t x[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      m = max(m, x[j] & 0x7FFFu);                 // |bf16| of the low element
      m = max(m, (x[j] >> 16) & 0x7FFFu);         // and of the high one
    }
  };
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  // four independent 16-byte loads in flight per thread, then the tail
  for (; i + 3 * stride < n8; i += 4 * stride) {
    uint4 w[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) w[u] = __ldg(src + i + u * stride);
#pragma unroll
    for (int u = 0; u < 4; ++u) fold(w[u]);
  }
  for (; i < n8; i += stride) fold(__ldg(src + i));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ uint32_t red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < 8; ++w) m = max(m, red[w]);
    grid_dep_wait();   // the zeroing of the output words is complete
    // bf16 bits << 16 are the FP32 bits of the same value
    atomicMax(reinterpret_cast<unsigned int*>(a.out) + blockIdx.y, m << 16);
  }
}

__global__ void zero_kernel(float* out) {
  grid_dep_launch();   // the maxima may start reading their inputs now
  if (threadIdx.x < 2) out[threadIdx.x] = 0.f;
}

__global__ void finalize_kernel(float* out) {
  grid_dep_wait();     // every block's maximum has landed
  const int i = threadIdx.x;
  if (i < 2) {
    const float amax = __uint_as_float(reinterpret_cast<const unsigned int*>(out)[i]);
    out[i] = (amax > 0.f) ? __fdiv_rn(amax, 2688.0f) : 1.0f;
  }
}

// Launched with programmatic stream serialisation after the one before it.
template <typename... P, typename... A>
static cudaError_t launch_pdl_calib(void (*k)(P...), dim3 grid, dim3 block, cudaStream_t st, A... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, args...);
}

// zero_kernel (an ordinary launch: it starts once everything before it on the
// stream, the inputs' producers included, has completed), then amax_kernel,
// which may start while the zeroing drains and reads its inputs before
// waiting for it, then finalize_kernel.
cudaError_t launch_calibrate(const CalibArgs& a, cudaStream_t st) {
  zero_kernel<<<1, 32, 0, st>>>(a.out);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (a.n > 0) {
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = (a.n / 8 + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sms) * 4;  // x 2 tensors: one wave of 8 blocks per SM
    const unsigned blocks = static_cast<unsigned>(want < cap ? (want > 0 ? want : 1) : cap);
    if ((e = launch_pdl_calib(amax_kernel, dim3(blocks, 2), dim3(256), st, a)) != cudaSuccess) return e;
  }
  return launch_pdl_calib(finalize_kernel, dim3(1), dim3(32), st, a.out);
}

}  // namespace kv4
