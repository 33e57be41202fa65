// Top-8 selection of one token's 256 router logits by one warp, shared by the decode paths.
#pragma once

#include "layer.cuh"

namespace moe {

// Order-preserving map of a float onto uint32 (larger float -> larger key).
__device__ __forceinline__ uint32_t float_key(float v) {
  const uint32_t u = __float_as_uint(v + 0.0f);  // -0 -> +0: equal floats get equal keys
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// (v, e) ranks above (w, f): larger value, or equal value and lower expert id.
__device__ __forceinline__ bool ranks_above(float v, int e, float w, int f) {
  return v > w || (v == w && e < f);
}

__device__ __forceinline__ void cas_pair(float& v0, int& i0, float& v1, int& i1) {
  const bool sw = ranks_above(v1, i1, v0, i0);
  const float a = sw ? v1 : v0, b = sw ? v0 : v1;
  const int ia = sw ? i1 : i0, ib = sw ? i0 : i1;
  v0 = a; v1 = b; i0 = ia; i1 = ib;
}

// Merges the descending list of the lane `o` apart (xor) into this lane's: the better of
// entry i and the partner's entry 7 - i keeps the top 8 of both as a bitonic sequence, which
// three half-cleaner stages sort.
__device__ __forceinline__ void top8_merge_xor(float (&v)[8], int (&id)[8], int o) {
  float w[8];
  int f[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    w[i] = __shfl_xor_sync(0xffffffffu, v[7 - i], o);
    f[i] = __shfl_xor_sync(0xffffffffu, id[7 - i], o);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const bool tk = ranks_above(w[i], f[i], v[i], id[i]);
    v[i] = tk ? w[i] : v[i];
    id[i] = tk ? f[i] : id[i];
  }
#pragma unroll
  for (int h = 4; h > 0; h >>= 1)
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if ((i & h) == 0) cas_pair(v[i], id[i], v[i + h], id[i + h]);
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
