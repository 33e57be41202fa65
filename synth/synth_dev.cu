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

__global__ void bytes_kernel(uint64_t key, uint64_t offset, uint64_t n, uint8_t* dst) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t j = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += stride) {
    uint64_t b = offset + j;
    dst[j] = (uint8_t)(fin(key + ((b >> 3) + 1) * kGamma) >> (8 * (b & 7)));
  }
}

__global__ void affine_kernel(uint64_t key, uint64_t offset, uint64_t n, float base,
                              uint16_t* scales, uint16_t* biases) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t j = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += stride) {
    uint32_t u = (uint32_t)(fin(key + (offset + j + 1) * kGamma) >> 41);
    float v = __fadd_rn(0.75f, __fmul_rn((float)u, 0x1p-24f));
    uint32_t w = __float_as_uint(__fmul_rn(v, base));
    w += 0x7FFFu + ((w >> 16) & 1u);
    uint16_t sb = (uint16_t)(w >> 16);
    scales[j] = sb;
    biases[j] = (uint16_t)((uint16_t)(sb ^ 0x8000u) + (uint16_t)(3u << 7));
  }
}

__global__ void uniform_kernel(uint64_t key, uint64_t offset, uint64_t n, float lo, float hi,
                               float* dst) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  const float span = __fsub_rn(hi, lo);
  for (uint64_t j = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += stride) {
    float u = __fmul_rn((float)(uint32_t)(fin(key + (offset + j + 1) * kGamma) >> 40), 0x1p-24f);
    dst[j] = __fadd_rn(lo, __fmul_rn(span, u));
  }
}

unsigned grid_for(uint64_t n) {
  uint64_t blocks = (n + 255) / 256;
  return (unsigned)(blocks > 152ull * 32 ? 152ull * 32 : blocks);
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

extern "C" int synth_bytes_device(uint64_t seed, uint64_t stream, uint64_t offset, uint64_t n,
                                  void* dst, void* cuda_stream) {
  if (n == 0) return 0;
  bytes_kernel<<<grid_for(n), 256, 0, (cudaStream_t)cuda_stream>>>(synth_key(seed, stream),
                                                                    offset, n, (uint8_t*)dst);
  return (int)cudaGetLastError();
}

extern "C" int synth_q4_affine_device(uint64_t seed, uint64_t stream, uint64_t offset, uint64_t n,
                                      float base, void* scales, void* biases, void* cuda_stream) {
  if (n == 0) return 0;
  affine_kernel<<<grid_for(n), 256, 0, (cudaStream_t)cuda_stream>>>(
      synth_key(seed, stream), offset, n, base, (uint16_t*)scales, (uint16_t*)biases);
  return (int)cudaGetLastError();
}

extern "C" int synth_uniform_f32_device(uint64_t seed, uint64_t stream, uint64_t offset,
                                        uint64_t n, float lo, float hi, void* dst,
                                        void* cuda_stream) {
  if (n == 0) return 0;
  uniform_kernel<<<grid_for(n), 256, 0, (cudaStream_t)cuda_stream>>>(
      synth_key(seed, stream), offset, n, lo, hi, (float*)dst);
  return (int)cudaGetLastError();
}
