// Device half of the seeded input generator: the same elements as synth_normal_bf16
// (definitions in synth.h), written straight into device memory.  Integer arithmetic and one
// fp32 multiply per element, so the bits equal the host generator's.
#include <cuda_runtime.h>
#include <stdint.h>

#include "synth.h"

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ULL;

__device__ __forceinline__ uint64_t fin(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

__device__ __forceinline__ uint16_t element(uint64_t key, uint64_t idx, float sigma) {
  int32_t s = 0;
#pragma unroll
  for (int w = 0; w < 3; ++w) {
    uint64_t v = fin(key + (3 * idx + (uint64_t)w + 1) * kGamma);
#pragma unroll
    for (int q = 0; q < 4; ++q) s += (int32_t)((v >> (16 * q)) & 0xFFFFu);
  }
  float z = __fmul_rn((float)(s - 393210), 0x1p-16f);
  uint32_t u = __float_as_uint(__fmul_rn(z, sigma));
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

__global__ void fill_kernel(uint64_t key, uint64_t offset, uint64_t n, float sigma, uint16_t* dst) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t j = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += stride)
    dst[j] = element(key, offset + j, sigma);
}

}  // namespace

extern "C" int synth_normal_bf16_device(uint64_t seed, uint64_t stream, uint64_t offset,
                                        uint64_t n, float sigma, void* dst, void* cuda_stream) {
  if (n == 0) return 0;
  uint64_t key = synth_key(seed, stream);
  uint64_t blocks = (n + 255) / 256;
  if (blocks > 152ull * 32) blocks = 152ull * 32;
  fill_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)cuda_stream>>>(key, offset, n, sigma,
                                                                      (uint16_t*)dst);
  return (int)cudaGetLastError();
}
