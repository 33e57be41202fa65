// A read-only HBM stream (measurement hook moe_read_probe in include/moe.h): every block
// reads its slice of the buffer with 16-byte non-caching loads, eight in flight per thread,
// and folds them into one word so that the loads cannot be dropped.  A pure read stream can
// run faster than the copy that the measured HBM peak comes from.
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"
#include "ptx.cuh"

namespace {

__global__ void __launch_bounds__(256) read_probe_kernel(const uint4* src, size_t n16,
                                                         uint32_t* sink) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  uint32_t acc = 0;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += 8 * stride) {
    uint4 v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (i + k * stride < n16) v[k] = moe::ld_stream_u4(src + i + k * stride);
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (i + k * stride < n16) acc ^= v[k].x ^ v[k].y ^ v[k].z ^ v[k].w;
  }
  if (acc == 0x9E3779B9u) *sink = acc;  // practically never: keeps the loads
}

}  // namespace

extern "C" int moe_read_probe(const void* buf, size_t bytes, void* sink, void* stream) {
  if (!buf || !sink || (bytes & 15) || (reinterpret_cast<uintptr_t>(buf) & 15) ||
      (reinterpret_cast<uintptr_t>(sink) & 3))
    return MOE_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};  // the launch's own status, not an earlier pending error
  cfg.gridDim = dim3(sms * 4);
  cfg.blockDim = dim3(256);
  cfg.stream = static_cast<cudaStream_t>(stream);
  return cudaLaunchKernelEx(&cfg, read_probe_kernel, static_cast<const uint4*>(buf),
                            (size_t)(bytes / 16), static_cast<uint32_t*>(sink)) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}
