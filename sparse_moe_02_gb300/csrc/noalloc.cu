// Routing of one token for callers that cannot allocate device memory.
//
// Every other entry point works on a handle whose workspace moe_create allocates with
// cudaMalloc.  Some callers cannot do that: a serving process whose device memory is
// reserved up front by another allocator (a KV-cache or activation pool that owns nearly
// all of HBM), or latency-critical code that may not call cudaMalloc, which can synchronise
// the whole device.  moe_route_one_noalloc gives them the routing of one token (router
// matrix-vector product, top 8, softmax weights) without a handle: its scratch -- the 256
// router logits and a block counter -- lives in the file-scope device array below, which
// every GPU that loads this library holds until the process exits.
//
// The array is shared by every call: calls whose kernels overlap on the GPU race on it (use
// one stream, or order the calls).  Its contents persist between calls; the counter, the
// only part that must start at zero, is cleared by each call before its kernel runs.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "layer.cuh"
#include "moe.h"
#include "ptx.cuh"

namespace moe {
namespace {

// Scratch: floats [0, 256) hold the logits, float slot 256 holds the block counter (int).
constexpr int kScratchFloats = kE + 64;  // 1,280 bytes
static __device__ __align__(256) float g_route_scratch[kScratchFloats];

constexpr int kNaWarps = 8;
constexpr int kNaBlocks = kE / kNaWarps;  // one router row per warp
constexpr int kMaxDevices = 64;

__device__ __forceinline__ float na_dot8(uint4 w, uint4 x) {
  const uint32_t a[4] = {w.x, w.y, w.z, w.w}, b[4] = {x.x, x.y, x.z, x.w};
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    s = fmaf(bf16_lo(a[i]), bf16_lo(b[i]), s);
    s = fmaf(bf16_hi(a[i]), bf16_hi(b[i]), s);
  }
  return s;
}

// The handle's selection rule with its own summation order: warp per router row, each lane
// keeping one fp32 running sum over its 16-byte chunks (lane l: chunks l, l + 32, ...), then a
// warp shuffle reduction.  The handle's batch-1 router sums each 256-chunk piece separately
// before adding the pieces, so for d > 2048 the two fp32 logits can differ in their last bits;
// the kept experts agree whenever the 8th and 9th logits are further apart than that rounding.
// The last block to finish keeps the 8 largest logits (ties: lower expert id) in ascending id
// with their softmax weights.
__global__ void __launch_bounds__(kNaWarps * 32)
    route_one_static_kernel(const __nv_bfloat16* x, int d, const __nv_bfloat16* w_r,
                            const float* bias, int32_t* topk_idx, float* topk_w, float* scratch) {
  extern __shared__ uint4 xs[];
  __shared__ int s_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nch = d / 8;
  const uint4* xsrc = reinterpret_cast<const uint4*>(x);
  for (int i = threadIdx.x; i < nch; i += blockDim.x) xs[i] = xsrc[i];
  __syncthreads();
  float* logits = scratch;
  int* counter = reinterpret_cast<int*>(scratch + kE);
  const int e = blockIdx.x * kNaWarps + warp;
  const __nv_bfloat16* row = w_r + (size_t)e * d;
  float acc = 0.f;
  for (int c = lane; c < nch; c += 32) acc += na_dot8(ld_stream_u4(row + (size_t)c * 8), xs[c]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) logits[e] = acc + (bias ? bias[e] : 0.f);
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(counter, 1) == (int)gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last || warp != 0) return;
  __threadfence();
  float v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __ldcg(logits + lane + 32 * i);
  uint32_t taken = 0;
  float wv[8];
  int wi[8];
#pragma unroll
  for (int r = 0; r < kTopK; ++r) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int id = lane + 32 * i;
      if (!((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && id < bi))) { bv = v[i]; bi = id; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    wv[r] = bv;
    wi[r] = bi;
  }
#pragma unroll
  for (int i = 0; i < 7; ++i)
#pragma unroll
    for (int j = 0; j < 7 - i; ++j)
      if (wi[j] > wi[j + 1]) {
        int ti = wi[j]; wi[j] = wi[j + 1]; wi[j + 1] = ti;
        float tv = wv[j]; wv[j] = wv[j + 1]; wv[j + 1] = tv;
      }
  float mx = wv[0];
#pragma unroll
  for (int j = 1; j < 8; ++j) mx = fmaxf(mx, wv[j]);
  float ex[8], s = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) { ex[j] = __expf(wv[j] - mx); s += ex[j]; }
  if (lane < kTopK) {
    int myi = wi[0];
    float myw = ex[0];
#pragma unroll
    for (int j = 1; j < 8; ++j)
      if (lane == j) { myi = wi[j]; myw = ex[j]; }
    topk_idx[lane] = myi;
    topk_w[lane] = myw / s;
  }
}

std::mutex g_setup_mu;
float* g_scratch_ptr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

// cuCtxGetCurrent through the runtime's driver entry point (the library does not link the
// driver library directly).
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  }
  return fn;
}

// Device address of the scratch array on device `dev` (which must be current): in host code
// the array's name is only a host-side stand-in.  The address is looked up with the device
// current and kept for that device's context; when the current context is a different one
// (after cudaDeviceReset the runtime creates a new primary context and loads the module again,
// so the array may have moved) it is looked up again.
cudaError_t scratch_for_device(int dev, float** out) {
  std::lock_guard<std::mutex> lock(g_setup_mu);
  const CtxGetCurrentFn get = ctx_get_current();
  if (!get) return cudaErrorInvalidDevice;
  // NULL before the runtime has made a context current on this thread
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS) return cudaErrorInvalidDevice;
  if (ctx && g_scratch_ptr[dev] && g_scratch_ctx[dev] == ctx) {
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
  }
  // the lookup itself makes the device's primary context current if none is
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_route_scratch);
  if (e != cudaSuccess) return e;
  if (get(&ctx) != CUDA_SUCCESS || !ctx) return cudaErrorInvalidDevice;
  g_scratch_ptr[dev] = static_cast<float*>(p);
  g_scratch_ctx[dev] = ctx;
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

extern "C" int moe_route_one_noalloc(const void* x, int d, const void* w_router,
                                     const float* router_bias, int32_t* topk_idx,
                                     float* topk_w, void* stream) {
  if (!x || !w_router || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
  if (d < 128 || d > 8192 || d % 128) return MOE_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w_router)) & 15u)
    return MOE_ERR_ALIGNMENT;
  if ((reinterpret_cast<uintptr_t>(router_bias) | reinterpret_cast<uintptr_t>(topk_idx) |
       reinterpret_cast<uintptr_t>(topk_w)) & 3u)
    return MOE_ERR_ALIGNMENT;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= moe::kMaxDevices)
    return MOE_ERR_CUDA;
  float* scratch = nullptr;
  if (moe::scratch_for_device(dev, &scratch) != cudaSuccess) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the block counter must start at zero
  if (cudaMemsetAsync(scratch + moe::kE, 0, sizeof(int), s) != cudaSuccess) return MOE_ERR_CUDA;
  // the launch's own status (not cudaGetLastError, which would also report and clear an
  // unrelated earlier error of the caller's)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(moe::kNaBlocks);
  cfg.blockDim = dim3(moe::kNaWarps * 32);
  cfg.dynamicSmemBytes = (size_t)d * 2;
  cfg.stream = s;
  const cudaError_t e = cudaLaunchKernelEx(
      &cfg, moe::route_one_static_kernel, static_cast<const __nv_bfloat16*>(x), d,
      static_cast<const __nv_bfloat16*>(w_router), router_bias, topk_idx, topk_w, scratch);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
