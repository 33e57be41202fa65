// Top-8 selection of one token's 256 router logits by one warp, shared by the decode paths.
#pragma once

#include "layer.cuh"

namespace moe {

// Order-preserving map of a float onto uint32 (larger float -> larger key).
__device__ __forceinline__ uint32_t float_key(float v) {
  const uint32_t u = __float_as_uint(v + 0.0f);  // -0 -> +0: equal floats get equal keys
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Warp-level selection from logits[256] (read through L2): the 8 largest (ties: lower id),
// listed in ascending expert id with their softmax weights; lanes 0..7 write ids[rank],
// w[rank].  Lane l holds the logits of ids l + 32 i.  Eight rounds, each taking the warp-wide
// largest remaining logit (redux max over order-preserving keys, then redux min over the ids
// holding it); the winners are then ranked by id.  The rounds stay a loop: the code runs
// once per launch from a cold instruction cache, where straight-line code is slow.
__device__ __forceinline__ void select_top8(const float* logits, int lane, int* ids, float* w) {
  float v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __ldcg(logits + lane + 32 * i);
  int my_id = 0;
  float my_v = 0.f;
  uint32_t taken = 0;  // bit i: id lane + 32 i already selected
#pragma unroll 1
  for (int r = 0; r < kTopK; ++r) {
    uint32_t bk = 0;
    int bid = 0x7fffffff;
    float bv = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t k = float_key(v[i]);
      // ids ascend with i: the first maximum in the lane wins ties
      if (!((taken >> i) & 1u) && (k > bk || bid == 0x7fffffff)) {
        bk = k;
        bid = lane + 32 * i;
        bv = v[i];
      }
    }
    const uint32_t best = __reduce_max_sync(0xffffffffu, bk);
    const int win = (int)__reduce_min_sync(0xffffffffu, bk == best ? (uint32_t)bid : 0xffffffffu);
    if (bid == win) taken |= 1u << (win >> 5);
    const float val = __shfl_sync(0xffffffffu, bv, win & 31);
    if (lane == r) {
      my_id = win;
      my_v = val;
    }
  }
  // lanes 0..7: softmax against the largest kept logit (the first winner), rank by id
  const float mx = __shfl_sync(0xffffffffu, my_v, 0);
  const float ex = lane < kTopK ? __expf(my_v - mx) : 0.f;
  float sum = ex;
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  int rank = 0;
#pragma unroll 1
  for (int k = 0; k < kTopK; ++k) rank += __shfl_sync(0xffffffffu, my_id, k) < my_id;
  if (lane < kTopK) {
    ids[rank] = my_id;
    w[rank] = ex / sum;
  }
}

}  // namespace moe
