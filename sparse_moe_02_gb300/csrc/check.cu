// Consistency check of a routing as moe_route writes it (include/moe.h, moe_check_routing):
//   topk_idx [T][8]: expert ids in [0, 256), strictly ascending within a token;
//   offsets [257]: offsets[0] = 0, non-decreasing, offsets[256] = 8T;
//   perm [8T]: slot s of group e (offsets[e] <= s < offsets[e + 1]) holds an entry p = t * 8 + j
//   with topk_idx[p] = e, strictly ascending within the group.
// Together these make perm a permutation of [0, 8T) whose groups are the experts' histogram in
// the stable order (§ "Keep expert routing on the GPU": histogram, prefix scan, scatter): a value
// p can only sit in group topk_idx[p], and at most once there.  Every value read is range-checked
// before it is used as an index, so arrays in any state give a status, never an access outside
// them.  The debug build (MOE_DEBUG) runs the same check inside every tensor-core forward and
// every moe_route, on the handle's own arrays, recording into the handle's device error word.
#include <cuda_runtime.h>
#include <stdint.h>

#include "layer.cuh"
#include "moe.h"
#include "ptx.cuh"

namespace moe {

namespace {

__global__ void check_routing_kernel(const int32_t* topk_idx, const int32_t* offsets,
                                     const int32_t* perm, int T, int* status) {
  const int n = T * kTopK;
  bool bad = false;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    bad = offsets[0] != 0 || offsets[kE] != n;
    for (int e = 0; e < kE; ++e) bad |= offsets[e + 1] < offsets[e];
  }
  const int stride = gridDim.x * blockDim.x;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    // entry i = t * 8 + j of topk_idx
    const int id = topk_idx[i];
    bad |= id < 0 || id >= kE;
    if (i % kTopK != 0) bad |= !(topk_idx[i - 1] < id);
    // slot i of perm: its group is the e with offsets[e] <= i < offsets[e + 1]
    const int p = perm[i];
    if (p < 0 || p >= n) {
      bad = true;
      continue;
    }
    int lo = 0, hi = kE;  // offsets[lo] <= i < offsets[hi] while the offsets are monotone
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (offsets[mid] <= i) lo = mid; else hi = mid;
    }
    const int e = lo, end = offsets[e + 1];
    bad |= !(offsets[e] <= i && i < end);
    bad |= topk_idx[p] != e;
    if (i + 1 < end && i + 1 < n) bad |= !(perm[i + 1] > p);
  }
  if (bad) atomicExch(status, kDevErrState);
}

}  // namespace

cudaError_t launch_check_routing(const int32_t* topk_idx, const int32_t* offsets,
                                 const int32_t* perm, int T, int* status, cudaStream_t s) {
  const int n = T * kTopK;
  const int blocks = n / 256 + 1 < 152 ? n / 256 + 1 : 152;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  return cudaLaunchKernelEx(&cfg, check_routing_kernel, topk_idx, offsets, perm, T, status);
}

}  // namespace moe

extern "C" int moe_check_routing(const int32_t* topk_idx, const int32_t* offsets,
                                 const int32_t* perm, int T, int* status, void* stream) {
  if (T < 0 || !status || (T > 0 && (!topk_idx || !perm)) || !offsets) return MOE_ERR_INVALID_ARG;
  if (T > (1 << 20)) return MOE_ERR_UNSUPPORTED;
  const uintptr_t m = reinterpret_cast<uintptr_t>(topk_idx) | reinterpret_cast<uintptr_t>(offsets) |
                      reinterpret_cast<uintptr_t>(perm) | reinterpret_cast<uintptr_t>(status);
  if (m & 3) return MOE_ERR_ALIGNMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(status, 0, sizeof(int), s) != cudaSuccess) return MOE_ERR_CUDA;
  return moe::launch_check_routing(topk_idx, offsets, perm, T, status, s) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}
