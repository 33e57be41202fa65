// Batch-1 decode of the MoE layer as matrix-vector products that stream only the selected
// experts' weights ("Optimizing on-device inference for Apple Silicon", § "Optimize the
// one-row weight path": a group of lanes cooperates on one output while reading different
// parts of the weight row; § "Reduce intermediate and state traffic": the two expert input
// projections run with their gated activation in one kernel, and the output projection
// with its routing score and the shared expert's result in another).
//
// Every weight row is read by one warp with 16-byte loads (lane l takes 16-byte chunks
// l, l+32, ...), multiplied by x (staged in shared memory) in fp32 and reduced with warp
// shuffles.  Three launches: (1) router rows + the shared expert's gate/up rows, with the
// top-8 selection done by the last router block to finish; (2) the 8 selected experts'
// gate/up rows; (3) the down rows of the 8 experts and the shared expert, weighted and
// summed in fixed order per output.
#include <algorithm>

#include <type_traits>

#include "layer.cuh"
#include "plan.cuh"
#include "ptx.cuh"
#include "select.cuh"
#include "q4.cuh"

namespace moe {
namespace {

constexpr int kWarps = 8;  // warps per block in every decode kernel
constexpr int kPre = 8;    // 16-byte chunks per lane held in registers per input row

__device__ __forceinline__ float dot8(uint4 w, uint4 x) {
  const uint32_t a[4] = {w.x, w.y, w.z, w.w}, b[4] = {x.x, x.y, x.z, x.w};
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    s = fmaf(bf16_lo(a[i]), bf16_lo(b[i]), s);
    s = fmaf(bf16_hi(a[i]), bf16_hi(b[i]), s);
  }
  return s;
}

// 8 bf16 weights times 8 fp32 values from shared memory.
__device__ __forceinline__ float dot8_f32(uint4 w, const float* h) {
  const float4 h0 = *reinterpret_cast<const float4*>(h);
  const float4 h1 = *reinterpret_cast<const float4*>(h + 4);
  float acc = bf16_lo(w.x) * h0.x;
  acc = fmaf(bf16_hi(w.x), h0.y, acc);
  acc = fmaf(bf16_lo(w.y), h0.z, acc);
  acc = fmaf(bf16_hi(w.y), h0.w, acc);
  acc = fmaf(bf16_lo(w.z), h1.x, acc);
  acc = fmaf(bf16_hi(w.z), h1.y, acc);
  acc = fmaf(bf16_lo(w.w), h1.z, acc);
  return fmaf(bf16_hi(w.w), h1.w, acc);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Up to kPre*32 16-byte chunks of one bf16 row, chunk c = base + lane + 32*i in v[i].
struct RowFrag {
  uint4 v[kPre];
};

__device__ __forceinline__ void row_load(RowFrag& r, const __nv_bfloat16* row, int nch, int lane,
                                         int base) {
#pragma unroll
  for (int i = 0; i < kPre; ++i) {
    const int c = base + lane + 32 * i;
    if (c < nch) r.v[i] = ld_stream_u4(row + (size_t)c * 8);
  }
}

__device__ __forceinline__ float row_dot(const RowFrag& r, const uint4* xs, int nch, int lane,
                                         int base) {
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < kPre; ++i) {
    const int c = base + lane + 32 * i;
    if (c < nch) acc += dot8(r.v[i], xs[c]);
  }
  return acc;
}

// Lane-partial dot product of a row with x; the first kPre*32 chunks are already in r.
__device__ __forceinline__ float row_dot_rest(RowFrag& r, const __nv_bfloat16* row,
                                              const uint4* xs, int nch, int lane) {
  float acc = row_dot(r, xs, nch, lane, 0);
  for (int base = kPre * 32; base < nch; base += kPre * 32) {
    row_load(r, row, nch, lane, base);
    acc += row_dot(r, xs, nch, lane, base);
  }
  return acc;
}

// Block-wide copy of n 16-byte words (read through L2) into shared memory, kDepth loads of a
// thread in flight before its stores: one round trip per batch instead of one per word.
template <int kDepth = 8>
__device__ __forceinline__ void stage_u4(const uint4* src, uint4* dst, int n) {
  for (int base = threadIdx.x; base < n; base += kDepth * blockDim.x) {
    uint4 v[kDepth];
#pragma unroll
    for (int i = 0; i < kDepth; ++i)
      if (base + i * (int)blockDim.x < n) v[i] = __ldcg(src + base + i * blockDim.x);
#pragma unroll
    for (int i = 0; i < kDepth; ++i)
      if (base + i * (int)blockDim.x < n) dst[base + i * blockDim.x] = v[i];
  }
}

// The whole block waits for the previous kernel on the stream, but only warp 0 executes
// griddepcontrol.wait: the other warps park on a hardware barrier, so that the waiting warps
// of the blocks that start early (beside the previous layer's blocks) take no issue slots from
// the blocks still working on the same SM.
__device__ __forceinline__ void pdl_wait_block() {
  if (threadIdx.x < 32) pdl_wait();
  __syncthreads();
}

__device__ __forceinline__ void stage_x(const __nv_bfloat16* x, uint4* xs, int d) {
  const uint4* src = reinterpret_cast<const uint4*>(x);
  for (int i = threadIdx.x; i < d / 8; i += blockDim.x) xs[i] = src[i];
  __syncthreads();
}

struct RouterSharedArgs {
  const __nv_bfloat16* x;
  DecodeWeights W;
  Dims D;
  int32_t *topk_idx, *offsets, *perm;
  float* topk_w;
  DecodeWs dw;
  int router_blocks;
  int* err;
};

// Blocks [0, router_blocks): one router row per warp, then the last block to finish selects
// the top 8.  Blocks after: one shared-expert feature (gate and up rows) per warp.  Weight
// rows are requested before waiting on the previous kernel (they do not depend on it).
// kShared: the launch also has the shared-expert blocks (a router-only launch keeps one row
// in registers per warp, small enough to stay resident beside the streamed decode launches).
template <bool kShared>
__global__ void __launch_bounds__(kWarps * 32) dec_router_shared_kernel(RouterSharedArgs a) {
  extern __shared__ uint4 xs[];
  __shared__ int s_last;
  __shared__ int s_ids[kTopK];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.D.d, nch = d / 8;
  const bool router = (int)blockIdx.x < a.router_blocks;
  const int c = ((int)blockIdx.x - a.router_blocks) * kWarps + warp;  // shared feature
  RowFrag r0, r1;
  if (router) {
    row_load(r0, a.W.w_r + (size_t)(blockIdx.x * kWarps + warp) * d, nch, lane, 0);
  } else if (kShared && c < a.D.fs) {
    row_load(r0, a.W.ws_gate + (size_t)c * d, nch, lane, 0);
    row_load(r1, a.W.ws_up + (size_t)c * d, nch, lane, 0);
  }
  pdl_trigger();    // the next launch only prefetches weights before its own wait
  pdl_wait_block();  // x may be written by the previous kernel
  // the streamed gate/up launch of this forward hands out work from this counter; every
  // launch that used it before has completed (the previous kernel on the stream has)
  if (blockIdx.x == 0 && threadIdx.x == 0) *a.dw.gu_next = 0;
  stage_x(a.x, xs, d);

  if (!router) {
    // shared expert: h_s[c] = silu(gate_c . x) * (up_c . x)
    if (kShared && c < a.D.fs) {
      const float g = warp_sum(row_dot_rest(r0, a.W.ws_gate + (size_t)c * d, xs, nch, lane));
      const float u = warp_sum(row_dot_rest(r1, a.W.ws_up + (size_t)c * d, xs, nch, lane));
      if (lane == 0) a.dw.hdec[(size_t)8 * a.D.hdim + c] = silu_mul(g, u);
    }
    return;
  }

  // router rows: logits[e] = w_r[e] . x (+ bias[e]); router_blocks * kWarps == E
  const int e = blockIdx.x * kWarps + warp;
  const float l = warp_sum(row_dot_rest(r0, a.W.w_r + (size_t)e * d, xs, nch, lane));
  if (lane == 0) a.dw.logits[e] = l + (a.W.bias ? a.W.bias[e] : 0.f);
  if (!a.topk_idx) return;  // the forward path selects in the next two kernels
  // routing outputs requested: the last router block to finish selects the top 8
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(a.dw.counter, 1) == a.router_blocks - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  __shared__ float s_w[kTopK];
  if (warp == 0) {
    select_top8(a.dw.logits, lane, s_ids, s_w);
    __syncwarp();
    if (lane < kTopK) {
      a.topk_idx[lane] = s_ids[lane];
      a.topk_w[lane] = s_w[lane];
      if (a.perm) a.perm[lane] = lane;  // one token: slot j holds assignment (0, j)
    }
    if (lane == 0) *a.dw.counter = 0;  // ready for the next launch on the stream
  }
  __syncthreads();
  if (a.offsets) {
    for (int e2 = threadIdx.x; e2 <= kE; e2 += blockDim.x) {
      int n = 0;
#pragma unroll
      for (int j = 0; j < kTopK; ++j) n += s_ids[j] < e2;
      a.offsets[e2] = n;
    }
  }
}

struct GateUpArgs {
  const __nv_bfloat16* x;
  DecodeWeights W;
  Dims D;
  int32_t* topk_idx;  // written by block 0 (the selection behind this forward)
  float* topk_w;
  DecodeWs dw;
};

// Items, one warp per item in a grid-stride loop over a grid that is fully resident: first
// the shared expert's features c < fs, then the selected experts' (j, c):
// h[j][c] = silu(gate . x) * (up . x).  A warp whose first item is a shared feature requests
// its rows before waiting on the router kernel (they do not depend on it).  Warp 0 of every
// block selects the top 8 from the router logits first.
__global__ void __launch_bounds__(kWarps * 32, 2) dec_gateup_kernel(GateUpArgs a) {
  extern __shared__ uint4 xs[];
  __shared__ int s_ids[kTopK];
  __shared__ float s_w[kTopK];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.D.d, f = a.D.f, fs = a.D.fs, nch = d / 8;
  const int total = fs + kTopK * f;
  const int nwarps = gridDim.x * kWarps;
  int it = blockIdx.x * kWarps + warp;
  RowFrag rg, ru;
  if (it < fs) {
    row_load(rg, a.W.ws_gate + (size_t)it * d, nch, lane, 0);
    row_load(ru, a.W.ws_up + (size_t)it * d, nch, lane, 0);
  }
  pdl_wait();     // the router logits come from the previous kernel
  pdl_trigger();  // the down kernel may start selecting and streaming its rows now
  if (warp == 0) select_top8(a.dw.logits, lane, s_ids, s_w);
  const uint4* src = reinterpret_cast<const uint4*>(a.x);
  for (int i = threadIdx.x; i < nch; i += blockDim.x) xs[i] = src[i];
  __syncthreads();
  if (blockIdx.x == 0 && threadIdx.x < kTopK) {
    a.topk_idx[threadIdx.x] = s_ids[threadIdx.x];
    a.topk_w[threadIdx.x] = s_w[threadIdx.x];
  }
  for (bool first = true; it < total; it += nwarps, first = false) {
    const __nv_bfloat16 *gr, *ur;
    size_t slot;
    if (it < fs) {  // the shared expert's feature it
      gr = a.W.ws_gate + (size_t)it * d;
      ur = a.W.ws_up + (size_t)it * d;
      slot = (size_t)8 * a.D.hdim + it;
    } else {
      const int j = (it - fs) / f, c = (it - fs) % f;
      const size_t row = ((size_t)s_ids[j] * f + c) * d;
      gr = a.W.w_gate + row;
      ur = a.W.w_up + row;
      slot = (size_t)j * a.D.hdim + c;
    }
    if (!(first && it < fs)) {  // the first shared item's rows are already in registers
      row_load(rg, gr, nch, lane, 0);
      row_load(ru, ur, nch, lane, 0);
    }
    const float g = warp_sum(row_dot_rest(rg, gr, xs, nch, lane));
    const float u = warp_sum(row_dot_rest(ru, ur, xs, nch, lane));
    if (lane == 0) a.dw.hdec[slot] = silu_mul(g, u);
  }
}

struct DownArgs {
  DecodeWeights W;
  Dims D;
  DecodeWs dw;
  __nv_bfloat16* y;
};

constexpr int kPreDown = 2;  // 16-byte chunks per lane held per down row (f <= 512 fully)

// One warp per output n (grid-stride over a fully resident grid): o_j = down_{e_j}[n] . h_j
// for the 8 experts and the shared expert; y[n] = bf16(sum_j w_j o_j (ascending expert id) +
// o_shared), accumulated in fp32.  The top 8 is selected again from the router logits (final:
// the router kernel completed before the gate/up kernel let this one start), so the down rows
// of the first output are requested before waiting for the gate/up kernel's h.
__global__ void __launch_bounds__(kWarps * 32, 2) dec_down_combine_kernel(DownArgs a) {
  extern __shared__ float hs[];  // [9][hdim]
  __shared__ int s_ids[kTopK];
  __shared__ float s_w[kTopK];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.D.d, f = a.D.f, fs = a.D.fs, hdim = a.D.hdim;
  if (warp == 0) select_top8(a.dw.logits, lane, s_ids, s_w);
  __syncthreads();
  const int nwarps = gridDim.x * kWarps;
  int n = blockIdx.x * kWarps + warp;
  uint4 pre[9][kPreDown];
  auto row_of = [&](int j, int nn) {
    return j < 8 ? a.W.w_down + ((size_t)s_ids[j] * d + nn) * f : a.W.ws_down + (size_t)nn * fs;
  };
  auto prefetch = [&](int nn) {
#pragma unroll
    for (int j = 0; j < 9; ++j) {
      const __nv_bfloat16* row = row_of(j, nn);
      const int nc = (j < 8 ? f : fs) / 8;
#pragma unroll
      for (int i = 0; i < kPreDown; ++i) {
        const int c = lane + 32 * i;
        if (c < nc) pre[j][i] = ld_stream_u4(row + (size_t)c * 8);
      }
    }
  };
  if (n < d) prefetch(n);
  pdl_wait();  // h comes from the gate/up kernel
  pdl_trigger();
  {
    // all loads of a batch are in flight before the first store (one L2 round trip per batch)
    const float4* src = reinterpret_cast<const float4*>(a.dw.hdec);
    float4* dst = reinterpret_cast<float4*>(hs);
    const int n4 = 9 * hdim / 4;
    for (int base = threadIdx.x; base < n4; base += 8 * blockDim.x) {
      float4 v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (base + i * (int)blockDim.x < n4) v[i] = __ldcg(src + base + i * blockDim.x);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (base + i * (int)blockDim.x < n4) dst[base + i * blockDim.x] = v[i];
    }
  }
  __syncthreads();
  for (; n < d; n += nwarps) {
    // per lane: sum over j (ascending expert id, then shared) of w_j * (its chunks of
    // down_j[n] . h_j); one warp reduction of those partials gives y[n] (fixed order)
    float y = 0.f;
#pragma unroll
    for (int j = 0; j < 9; ++j) {
      const int nc = (j < 8 ? f : fs) / 8;
      const float* hj = hs + (size_t)j * hdim;
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < kPreDown; ++i) {
        const int c = lane + 32 * i;
        if (c < nc) acc += dot8_f32(pre[j][i], hj + c * 8);
      }
      const __nv_bfloat16* row = row_of(j, n);
      for (int c = lane + 32 * kPreDown; c < nc; c += 32)
        acc += dot8_f32(ld_stream_u4(row + (size_t)c * 8), hj + c * 8);
      y = fmaf(j < 8 ? s_w[j] : 1.0f, acc, y);
    }
    y = warp_sum(y);
    if (lane == 0) a.y[n] = __float2bfloat16_rn(y);
    if (n + nwarps < d) prefetch(n + nwarps);
  }
}

// ---------------------------------------------------------------- small batches (2..8 tokens)
//
// The speculative-verify shape (§ "Limits of further optimization": verifying a few draft
// tokens at once): each token keeps its own top 8, and every weight row of the union of the
// selected experts is read once and applied to every token that chose that expert.  Per token
// the sum keeps the single-token order: ascending expert id, then the shared expert.

// Lane-partial dot products of one d-element row with the x rows of the tokens in `mask`
// (bit t: token t, at xs + t * nch), kPre*32 pieces at a time; the first such piece group is
// already in r.  mask is the same in every lane.
template <int NT>
__device__ __forceinline__ void row_dot_tokens(RowFrag& r, const __nv_bfloat16* row,
                                               const uint4* xs, int nch, int mask, int lane,
                                               float (&acc)[NT]) {
  for (int base = 0; base < nch; base += kPre * 32) {
    if (base) row_load(r, row, nch, lane, base);
#pragma unroll
    for (int t = 0; t < NT; ++t)
      if ((mask >> t) & 1) acc[t] += row_dot(r, xs + (size_t)t * nch, nch, lane, base);
  }
}

// Per-block view of the batch's routing: each token's top 8 (ascending id) and weights, and
// the union of the selections in ascending expert id with, per expert, the mask of tokens
// that chose it.
struct BatchSel {
  int ids[kGemvMaxTokens][kTopK];
  float w[kGemvMaxTokens][kTopK];
  int tmask[kE];
  int ulist[kE];
  int nu;
};

// Every thread of the block calls this (it holds barriers); logits [T][E] read through L2.
__device__ void batch_select(const float* logits, int T, BatchSel& S) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < kE; e += blockDim.x) S.tmask[e] = 0;
  if (warp < T) select_top8(logits + (size_t)warp * kE, lane, S.ids[warp], S.w[warp]);
  __syncthreads();
  if ((int)threadIdx.x < T * kTopK)
    atomicOr(&S.tmask[S.ids[threadIdx.x / kTopK][threadIdx.x % kTopK]], 1 << (threadIdx.x / kTopK));
  __syncthreads();
  if (warp == 0) {
    int n = 0;
    for (int e0 = 0; e0 < kE; e0 += 32) {
      const bool used = S.tmask[e0 + lane] != 0;
      const uint32_t bal = __ballot_sync(0xffffffffu, used);
      if (used) S.ulist[n + __popc(bal & ((1u << lane) - 1u))] = e0 + lane;
      n += __popc(bal);
    }
    if (lane == 0) S.nu = n;
  }
  __syncthreads();
}

// Position of expert e in token t's top 8 (e was selected by t).
__device__ __forceinline__ int batch_slot(const BatchSel& S, int t, int e) {
  int j = 0;
#pragma unroll
  for (int i = 0; i < kTopK; ++i) j = S.ids[t][i] == e ? i : j;
  return j;
}

struct BatchRouterArgs {
  const __nv_bfloat16* x;
  DecodeWeights W;
  Dims D;
  int T;
  int32_t *topk_idx, *offsets, *perm;  // routing outputs (NULL topk_idx: forward)
  float* topk_w;
  DecodeWs dw;
  int router_blocks;
  bool plan;      // routing for the tensor-core schedule: the last block also builds the plan
  PlanArgs pa;    // (offsets, group starts, unit lists) in rws and scatters the tokens,
  RouteWs rws;    // perm included, so that no separate plan launch follows
};

// Blocks [0, router_blocks): one router row per warp for all T tokens; in a routing-only
// launch the last block to finish selects and writes topk_idx / topk_w / offsets / perm.
// Blocks after: one shared-expert feature per warp, h_s[t][c] for every token.
// Instantiated per token count TT (= a.T), as the gate/up and down kernels below.
template <int TT>
__global__ void __launch_bounds__(kWarps * 32) dec_batch_router_shared_kernel(BatchRouterArgs a) {
  extern __shared__ uint4 xs[];  // [T][d/8]
  __shared__ int s_last;
  __shared__ BatchSel S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.D.d, nch = d / 8, T = TT;
  const bool router = (int)blockIdx.x < a.router_blocks;
  const int c = ((int)blockIdx.x - a.router_blocks) * kWarps + warp;
  RowFrag r0, r1;
  if (router) {
    row_load(r0, a.W.w_r + (size_t)(blockIdx.x * kWarps + warp) * d, nch, lane, 0);
  } else if (c < a.D.fs) {
    row_load(r0, a.W.ws_gate + (size_t)c * d, nch, lane, 0);
    row_load(r1, a.W.ws_up + (size_t)c * d, nch, lane, 0);
  }
  pdl_wait();  // x may be written by the previous kernel
  pdl_trigger();
  stage_u4(reinterpret_cast<const uint4*>(a.x), xs, T * nch);
  __syncthreads();
  if (!router) {
    if (c < a.D.fs) {
      float g[TT], u[TT];
#pragma unroll
      for (int t = 0; t < TT; ++t) g[t] = u[t] = 0.f;
      row_dot_tokens(r0, a.W.ws_gate + (size_t)c * d, xs, nch, (1 << T) - 1, lane, g);
      row_dot_tokens(r1, a.W.ws_up + (size_t)c * d, xs, nch, (1 << T) - 1, lane, u);
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        const float gv = warp_sum(g[t]), uv = warp_sum(u[t]);
        if (lane == 0) a.dw.hdec[((size_t)t * 9 + 8) * a.D.hdim + c] = silu_mul(gv, uv);
      }
    }
    return;
  }
  const int e = blockIdx.x * kWarps + warp;
  float l[TT];
#pragma unroll
  for (int t = 0; t < TT; ++t) l[t] = 0.f;
  row_dot_tokens(r0, a.W.w_r + (size_t)e * d, xs, nch, (1 << T) - 1, lane, l);
#pragma unroll
  for (int t = 0; t < TT; ++t) {
    const float v = warp_sum(l[t]);
    if (lane == 0) a.dw.logits[(size_t)t * kE + e] = v + (a.W.bias ? a.W.bias[e] : 0.f);
  }
  if (!a.topk_idx) return;  // the forward path selects in the next two kernels
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(a.dw.counter, 1) == a.router_blocks - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  batch_select(a.dw.logits, T, S);
  if (a.plan) {
    // the plan of the tensor-core schedule (one token block): per-expert counts, groups,
    // unit lists, and the scatter of the T tokens (it reads topk_idx as written here)
    __shared__ GroupTable G;
    __shared__ int s_pre[kE];
    __shared__ uint32_t mask[4][kE];
    if ((int)threadIdx.x < T * kTopK) {
      const int t = threadIdx.x / kTopK, j = threadIdx.x % kTopK;
      a.topk_idx[t * kTopK + j] = S.ids[t][j];
      a.topk_w[t * kTopK + j] = S.w[t][j];
    }
    for (int i = threadIdx.x; i < 4 * kE; i += blockDim.x) (&mask[0][0])[i] = 0u;
    const int e2 = threadIdx.x;  // 256 threads: one per expert
    int cnt = 0;
    for (int i = 0; i < T * kTopK; ++i) cnt += S.ids[i / kTopK][i % kTopK] == e2;
    s_pre[e2] = 0;
    plan_groups(a.pa, cnt, G, a.rws, true);  // ends with a barrier
    plan_units(G, a.rws.units_gu, false, 0, G.n_gu, T);
    plan_units(G, a.rws.units_dn, true, 0, G.n_dn, T);
    scatter_block(0, T, a.topk_idx, a.perm, a.rws, mask, s_pre, G.off, G.poff, G.p_shared);
    if (threadIdx.x == 0) *a.dw.counter = 0;  // ready for the next launch on the stream
    return;
  }
  if ((int)threadIdx.x < T * kTopK) {
    const int t = threadIdx.x / kTopK, j = threadIdx.x % kTopK, id = S.ids[t][j];
    a.topk_idx[t * kTopK + j] = id;
    a.topk_w[t * kTopK + j] = S.w[t][j];
    // slot of (t, j): assignments grouped by expert, tokens ascending within a group
    int rank = 0;
    for (int t2 = 0; t2 < T; ++t2)
      for (int j2 = 0; j2 < kTopK; ++j2) {
        const int id2 = S.ids[t2][j2];
        rank += id2 < id || (id2 == id && t2 < t);
      }
    if (a.perm) a.perm[rank] = t * kTopK + j;
  }
  if (a.offsets)
    for (int e2 = threadIdx.x; e2 <= kE; e2 += blockDim.x) {
      int n = 0;
      for (int i = 0; i < T * kTopK; ++i) n += S.ids[i / kTopK][i % kTopK] < e2;
      a.offsets[e2] = n;
    }

  if (threadIdx.x == 0) *a.dw.counter = 0;  // ready for the next launch on the stream
}

struct BatchGateUpArgs {
  const __nv_bfloat16* x;
  DecodeWeights W;
  Dims D;
  int T;
  int32_t* topk_idx;  // written by block 0 (the selection behind this forward)
  float* topk_w;
  DecodeWs dw;
};

// Items (union expert k, feature c), one warp per item over a resident grid: the gate and up
// rows are read once; h[t][slot][c] = silu(gate . x_t) * (up . x_t) for every token t that
// chose the expert.
// Instantiated per token count TT (= a.T): the per-token loops unroll TT times, so a small
// batch runs a small body (unrolled for the largest batch, the code missed in the instruction
// cache).
template <int TT>
__global__ void __launch_bounds__(kWarps * 32, 2) dec_batch_gateup_kernel(BatchGateUpArgs a) {
  extern __shared__ uint4 xs[];  // [T][d/8]
  __shared__ BatchSel S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.D.d, f = a.D.f, nch = d / 8, T = TT;
  pdl_wait();     // the router logits come from the previous kernel
  pdl_trigger();  // the down kernel may start selecting and streaming its rows now
  batch_select(a.dw.logits, T, S);
  stage_u4(reinterpret_cast<const uint4*>(a.x), xs, T * nch);
  if (blockIdx.x == 0 && (int)threadIdx.x < T * kTopK) {
    a.topk_idx[threadIdx.x] = S.ids[threadIdx.x / kTopK][threadIdx.x % kTopK];
    a.topk_w[threadIdx.x] = S.w[threadIdx.x / kTopK][threadIdx.x % kTopK];
  }
  __syncthreads();
  const int nwarps = gridDim.x * kWarps, items = S.nu * f;
  for (int it = blockIdx.x * kWarps + warp; it < items; it += nwarps) {
    const int k = it / f, c = it % f, e = S.ulist[k], mask = S.tmask[e];
    const size_t row = ((size_t)e * f + c) * d;
    RowFrag rg, ru;
    row_load(rg, a.W.w_gate + row, nch, lane, 0);
    row_load(ru, a.W.w_up + row, nch, lane, 0);
    float g[TT], u[TT];
#pragma unroll
    for (int t = 0; t < TT; ++t) g[t] = u[t] = 0.f;
    row_dot_tokens(rg, a.W.w_gate + row, xs, nch, mask, lane, g);
    row_dot_tokens(ru, a.W.w_up + row, xs, nch, mask, lane, u);
#pragma unroll
    for (int t = 0; t < TT; ++t)
      if ((mask >> t) & 1) {
        const float gv = warp_sum(g[t]), uv = warp_sum(u[t]);
        if (lane == 0)
          a.dw.hdec[((size_t)t * 9 + batch_slot(S, t, e)) * a.D.hdim + c] = silu_mul(gv, uv);
      }
  }
}

struct BatchDownArgs {
  DecodeWeights W;
  Dims D;
  int T;
  DecodeWs dw;
  __nv_bfloat16* y;
};

constexpr int kBatchRows = 8;  // union experts whose down rows one warp has in flight at once

// One warp per output n over a resident grid: the down rows of the union experts, eight at a
// time (the first eight requested before waiting for h), each applied to the tokens that
// chose it; per lane and token the terms w_tj (down_e[n] . h_tj) add in ascending expert id,
// then the shared expert's; one warp reduction per token gives y[t][n].
template <int TT>
__global__ void __launch_bounds__(kWarps * 32, 2) dec_batch_down_combine_kernel(BatchDownArgs a) {
  extern __shared__ float hs[];  // [T][9][hdim]
  __shared__ BatchSel S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.D.d, f = a.D.f, fs = a.D.fs, hdim = a.D.hdim, T = TT;
  const int nc = f / 8;
  batch_select(a.dw.logits, T, S);  // final: the router finished before this launch started
  const int nwarps = gridDim.x * kWarps;
  int n = blockIdx.x * kWarps + warp;
  uint4 pre[kBatchRows][kPreDown];
  auto load_group = [&](int k0, int nn) {
#pragma unroll
    for (int q = 0; q < kBatchRows; ++q)
      if (k0 + q < S.nu) {
        const __nv_bfloat16* row = a.W.w_down + ((size_t)S.ulist[k0 + q] * d + nn) * f;
#pragma unroll
        for (int i = 0; i < kPreDown; ++i)
          if (lane + 32 * i < nc) pre[q][i] = ld_stream_u4(row + (size_t)(lane + 32 * i) * 8);
      }
  };
  if (n < d) load_group(0, n);
  pdl_wait();  // h comes from the gate/up kernel
  pdl_trigger();
  // four deep: the rows prefetched before the wait are live in registers meanwhile
  stage_u4<4>(reinterpret_cast<const uint4*>(a.dw.hdec), reinterpret_cast<uint4*>(hs),
              T * 9 * hdim / 4);
  __syncthreads();
  for (; n < d; n += nwarps) {
    float acc[TT];
#pragma unroll
    for (int t = 0; t < TT; ++t) acc[t] = 0.f;
    for (int k0 = 0; k0 < S.nu; k0 += kBatchRows) {
      if (k0) load_group(k0, n);
#pragma unroll
      for (int q = 0; q < kBatchRows; ++q) {
        if (k0 + q >= S.nu) break;
        const int e = S.ulist[k0 + q], mask = S.tmask[e];
        const __nv_bfloat16* row = a.W.w_down + ((size_t)e * d + n) * f;
#pragma unroll
        for (int t = 0; t < TT; ++t)
          if (t < T && ((mask >> t) & 1)) {
            const int j = batch_slot(S, t, e);
            const float* ht = hs + ((size_t)t * 9 + j) * hdim;
            float sj = 0.f;
#pragma unroll
            for (int i = 0; i < kPreDown; ++i) {
              const int cc = lane + 32 * i;
              if (cc < nc) sj += dot8_f32(pre[q][i], ht + cc * 8);
            }
            for (int cc = lane + 32 * kPreDown; cc < nc; cc += 32)
              sj += dot8_f32(ld_stream_u4(row + (size_t)cc * 8), ht + cc * 8);
            acc[t] = fmaf(S.w[t][j], sj, acc[t]);
          }
      }
    }
    // the shared expert, weight 1
    const __nv_bfloat16* srow = a.W.ws_down + (size_t)n * fs;
    for (int cc = lane; cc < fs / 8; cc += 32) {
      const uint4 wv = ld_stream_u4(srow + (size_t)cc * 8);
#pragma unroll
      for (int t = 0; t < TT; ++t)
        if (t < T) acc[t] += dot8_f32(wv, hs + ((size_t)t * 9 + 8) * hdim + cc * 8);
    }
#pragma unroll
    for (int t = 0; t < TT; ++t)
      if (t < T) {
        const float v = warp_sum(acc[t]);
        if (lane == 0) a.y[(size_t)t * d + n] = __float2bfloat16_rn(v);
      }
    if (n + nwarps < d) load_group(0, n + nwarps);
  }
}

// ---------------------------------------------------------------- streamed batch-1 decode
//
// The layer's expert work after the router as one launch of one block per SM (§ "Optimize the
// one-row weight path": the one-row path is bound by reading weights; § "Reduce intermediate
// and state traffic": the gated activation is fused with the input projections, and the
// routing scores and the shared expert with the output projection).  A block takes about
// 212 KB of shared memory at d = 2048, f = 512, so exactly one runs on every SM:
//   - warp 0 selects the top 8 once the router launch has finished and copies the block's slice
//     of down rows -- outputs [n0, n1) of the 8 experts and of the shared expert, about 126 KB
//     -- into shared memory, the routed ones while the slot warps fetch their last items;
//   - the block's gate/up items are every G-th feature (the shared expert's, then the selected
//     experts'); each of eight further warps owns one ring slot (one feature's gate and up
//     rows), takes the block's next item whenever its slot is free, refills the slot by bulk
//     asynchronous copies, takes the dot products with x and writes
//     h = silu(gate . x) * (up . x) (fp32) to global memory; items are requested into L2 two
//     rounds ahead of their copy (HBM needs about 20 MB in flight over the chip to run at full
//     rate, far more than the ring holds);
//   - the blocks then meet at a grid-wide barrier (a counter the router launch zeroes; the
//     launch's blocks are all resident, one per SM, once the previous layer's have left), load
//     all of h and combine their outputs in fixed order.
// Shapes whose buffers do not fit use dec_gateup / dec_down_combine above.

constexpr int kStSlots = 8;                    // ring slots: one feature's gate and up rows each
constexpr int kStThreads = 32 * (1 + kStSlots);  // warp 0 + one warp per slot
constexpr int kCbWarps = kStSlots;             // the slot warps also run the combine
constexpr int kStMaxOut = 16;                  // outputs per block: four per output group
constexpr int kDownLead = 12;                  // gate/up items left when the down rows go out

struct StreamArgs {
  const __nv_bfloat16* x;
  DecodeWeights W;    // the router; the experts of a bf16 launch
  Q4Weights Q;        // the experts of a 4-bit launch
  Dims D;
  int32_t* topk_idx;  // written by block 0 (the selection behind this forward)
  float* topk_w;
  DecodeWs dw;
  __nv_bfloat16* y;
  int* err;
  int bar_extra;      // arrivals the grid barrier waits for beyond the launch's blocks (0)
  uint64_t limit_ns;  // how long the grid barrier waits before it reports a timeout
};

// Shared-memory layout of a block, in bytes: the ring (kStSlots slots of one feature's gate and
// up rows, two per slot warp with 4-bit rows), x, the down rows of up to nn = ceil(d / G) outputs of the 8 experts and the shared
// expert, h, the mbarriers.  bf16: x as bf16, h as two fp32 planes (see h_piece).  4-bit: a
// slot holds the two rows' codes, then their scales and biases; x as swizzled fp32 with its sums
// per 32, h as swizzled fp32 (see q4.cuh); the down rows as codes [9][nn][K/2], then scales, then biases
// (K = f, or fs for the shared expert).  A 4-bit block is padded to more than half an SM's
// shared memory, so that one block runs on every SM.
struct StLayout {
  uint32_t slot, xs, xsum, rows, sc, bi, hp, hsum, bars, total;
};
template <bool Q4>
__host__ __device__ inline StLayout st_layout(const Dims& D, int G) {
  StLayout L;
  const int nn = (D.d + G - 1) / G;
  if (!Q4) {
    L.slot = 4 * D.d;
    L.xs = kStSlots * L.slot;
    L.xsum = L.rows = L.xs + 2 * D.d;
    L.sc = L.bi = L.hp = L.rows + round_up(nn * (8 * D.f + D.fs) * 2, 16);
    L.hsum = L.bars = L.hp + 9 * D.hdim * 4;
  } else {
    L.slot = D.d + D.d / 8;  // codes d/2 each, scales and biases d/32 bytes each
    L.xs = 2 * kStSlots * L.slot;  // two slots per slot warp
    L.xsum = L.xs + 4 * D.d;
    L.rows = L.xsum + 4 * (D.d / 32);
    L.sc = L.rows + nn * (8 * D.f + D.fs) / 2;
    L.bi = L.sc + nn * (8 * D.f + D.fs) / 32;
    L.hp = L.bi + nn * (8 * D.f + D.fs) / 32;
    L.hsum = L.bars = L.hp + 9 * D.hdim * 4;
  }
  L.total = L.bars + (2 * kStSlots + 2) * 8;
  if (Q4 && L.total < 120 * 1024) L.total = 120 * 1024;
  return L;
}

// 8 bf16 weights times 8 fp32 values.
__device__ __forceinline__ float dot8_f32v(uint4 w, float4 h0, float4 h1) {
  float a = bf16_lo(w.x) * h0.x, b = bf16_hi(w.x) * h0.y;
  a = fmaf(bf16_lo(w.y), h0.z, a);
  b = fmaf(bf16_hi(w.y), h0.w, b);
  a = fmaf(bf16_lo(w.z), h1.x, a);
  b = fmaf(bf16_hi(w.z), h1.y, b);
  a = fmaf(bf16_lo(w.w), h1.z, a);
  b = fmaf(bf16_hi(w.w), h1.w, b);
  return a + b;
}

// The h vectors in shared memory as two planes: plane q holds floats 4q .. 4q + 3 of every
// 8-float piece, piece c of expert rank j (j = 8: the shared expert) at float4 index
// j * hdim / 8 + c of its plane -- so that 32 lanes reading 32 consecutive pieces read 512
// contiguous bytes per load (no bank conflict), against 32-byte strides in the plain layout.
__device__ __forceinline__ float4 h_piece(const float4* hp, int hdim, int j, int c, int q) {
  return hp[(size_t)q * (9 * hdim / 8) + (size_t)j * (hdim / 8) + c];
}

// out[i] = bf16(sum_j w_j (rows_j[i] . h_j) + rows_s[i] . h_s) for i < nn (1 <= nn <= 16), by
// the kCbWarps warps of the combine (cw: this warp's index among them, ct: this thread's): the
// rows of expert rank j at rows + j nn 2f, the shared expert's at rows + 8 nn 2f (2fs bytes
// each).  Combine warp w takes the outputs w % 4, w % 4 + 4, ... and half w / 4 of every row's
// 16-byte pieces, lane l the pieces l, l + 32, ... of that half: each row byte and each h byte
// is read once per warp that needs it, in 512-byte conflict-free loads.  Per output and piece
// the terms run over the experts in ascending id, then the shared expert; pieces within a lane,
// then lanes, then the two halves are added after.  All combine threads call this (it holds
// named barrier 4); part is shared scratch of kCbWarps * 4 floats.
__device__ __forceinline__ void dn_combine_rows(const uint8_t* rows, const float4* hp, int nn,
                                                int f, int fs, int hdim, const float* w,
                                                float* part, __nv_bfloat16* out, int cw,
                                                int ct) {
  const int lane = ct & 31;
  const int og = cw & 3, half = cw >> 2;
  const size_t rb = (size_t)f * 2, srb = (size_t)fs * 2;
  // the four outputs of this warp; past nn the last row is read again and its sum dropped, so
  // that the loop body has no branch (a branch per output keeps the compiler from interleaving
  // the outputs' dot products, and the warp then stalls on each short chain)
  int oi[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) oi[m] = min(og + 4 * m, nn - 1);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  auto piece = [&](int j, int c, const uint8_t* base, size_t pitch, float wj) {
    const float4 ha = h_piece(hp, hdim, j, c, 0), hb = h_piece(hp, hdim, j, c, 1);
#pragma unroll
    for (int m = 0; m < 4; ++m)
      acc[m] = fmaf(wj, dot8_f32v(reinterpret_cast<const uint4*>(base + oi[m] * pitch)[c], ha, hb),
                    acc[m]);
  };
  if (f == fs && f % 512 == 0) {
    // one row length, a whole number of pieces per lane: pieces outer, the 9 experts unrolled
    // inside (straight-line code over all of them)
    const int K8 = f / 8;
    for (int c = half * K8 / 2 + lane; c < (half + 1) * K8 / 2; c += 32) {
#pragma unroll
      for (int j = 0; j < 9; ++j) piece(j, c, rows + j * nn * rb, rb, j < 8 ? w[j] : 1.0f);
    }
  } else {
#pragma unroll 1
    for (int j = 0; j < 9; ++j) {
      const int K8 = (j < 8 ? f : fs) / 8;
      const uint8_t* base = rows + (j < 8 ? j * nn * rb : 8 * nn * rb);
      const size_t pitch = j < 8 ? rb : srb;
      const float wj = j < 8 ? w[j] : 1.0f;
      for (int c = half * K8 / 2 + lane; c < (half + 1) * K8 / 2; c += 32)
        piece(j, c, base, pitch, wj);
    }
  }
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const float v = warp_sum(acc[m]);
    if (lane == 0) part[cw * 4 + m] = v;
  }
  named_sync(4, kCbWarps * 32);
  if (ct < nn) {
    const int g = ct & 3, m = ct >> 2;
    out[ct] = __float2bfloat16_rn(part[g * 4 + m] + part[(g + 4) * 4 + m]);
  }
}
static_assert(kCbWarps == 8, "the combine pairs warps w and w + 4 (two halves of K)");

// Stages v (n bf16 values, n a multiple of 32) as swizzled fp32 in vf and the sums of each 32 in
// vs, by the nthreads threads of named barrier `bar` (thread index t); ends with that barrier.
__device__ __forceinline__ void stage_f32_named(const __nv_bfloat16* src, float* vf, float* vs,
                                                int n, int t, int nthreads, int bar) {
  const uint4* s16 = reinterpret_cast<const uint4*>(src);
  for (int m = t; m < n / 8; m += nthreads) {
    const uint4 v = __ldcg(s16 + m);
    *reinterpret_cast<float4*>(vf + swz(8 * m)) =
        make_float4(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y));
    *reinterpret_cast<float4*>(vf + swz(8 * m + 4)) =
        make_float4(bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w));
  }
  named_sync(bar, nthreads);
  // a piece's 32 values are its 32 slots in some order: summed in slot order
  for (int p = t; p < n / 32; p += nthreads) {
    const float4* q = reinterpret_cast<const float4*>(vf + 32 * p);
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 u = q[i];
      sum += u.x;
      sum += u.y;
      sum += u.z;
      sum += u.w;
    }
    vs[p] = sum;
  }
  named_sync(bar, nthreads);
}

__device__ __forceinline__ float bf16_at(const uint8_t* p) {
  return __uint_as_float((uint32_t)*reinterpret_cast<const unsigned short*>(p) << 16);
}

// The 4-bit combine: out[i] for i < nn (1 <= nn <= 16) over the rows in shared memory (codes
// [9][nn][K/2], then scales and biases [9][nn][K/64] bf16, K = f, or fs for the shared expert;
// layout in st_layout) and h (swizzled rows at hf + j hdim), by the kCbWarps warps of the combine
// (cw: this warp's index among them, ct: this thread's).  The 32-input pieces of the nine rows
// are taken as one run (P < 8 f / 32: routed row j = P / (f / 32); then the shared row); combine
// warp w takes the outputs w % 4, w % 4 + 4, ... and half w / 4 of the run, lane l the pieces
// l, l + 32, ... of that half.  A piece of h and its sum are read once and applied to the
// warp's four outputs, each term w_j (scale * (codes . h_j) + bias * sum h_j); the two halves
// are added after.  All combine threads call this (it holds named barrier 4); part is shared
// scratch of kCbWarps * 4 floats.
__device__ __forceinline__ void dn_combine_q4(const uint8_t* codes, const uint8_t* sc,
                                              const uint8_t* bi, const float* hf, int nn, int f,
                                              int fs, int hdim, const float* w, float* part,
                                              __nv_bfloat16* out, int cw, int ct) {
  const int lane = ct & 31;
  const int og = cw & 3, half = cw >> 2;
  const int npr = f / 32, npt = 8 * npr + fs / 32;
  // past nn the last row is read again and its sum dropped (no branch per output)
  int oi[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) oi[m] = min(og + 4 * m, nn - 1);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const int p1 = half ? npt : npt / 2;
  for (int P = (half ? npt / 2 : 0) + lane; P < p1; P += 32) {
    const int j = P < 8 * npr ? P / npr : 8, p = P - j * npr;
    float4 hv[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) hv[k] = piece_f4(hf + (size_t)j * hdim, p, k);
    float hsum = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) hsum += (hv[k].x + hv[k].y) + (hv[k].z + hv[k].w);
    const float wj = j < 8 ? w[j] : 1.0f;
    // the row's codes and its scales / biases (bytes) in their regions
    const size_t kb = j < 8 ? (size_t)f / 2 : (size_t)fs / 2;    // code bytes of a row
    const size_t gbr = j < 8 ? (size_t)f / 32 : (size_t)fs / 32;  // scale bytes of a row
    const size_t cbase = j < 8 ? (size_t)j * nn * (f / 2) : (size_t)8 * nn * (f / 2);
    const size_t gbase = j < 8 ? (size_t)j * nn * (f / 32) : (size_t)8 * nn * (f / 32);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const uint4 c = *reinterpret_cast<const uint4*>(codes + cbase + oi[m] * kb + (size_t)p * 16);
      const size_t g = gbase + oi[m] * gbr + (p / 2) * 2;
      const float t = bf16_at(sc + g) * q4_dot32(c, hv) + bf16_at(bi + g) * hsum;
      acc[m] = fmaf(wj, t, acc[m]);
    }
  }
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const float v = warp_sum(acc[m]);
    if (lane == 0) part[cw * 4 + m] = v;
  }
  named_sync(4, kCbWarps * 32);
  if (ct < nn) {
    const int g = ct & 3, m = ct >> 2;
    out[ct] = __float2bfloat16_rn(part[g * 4 + m] + part[(g + 4) * 4 + m]);
  }
}

// At most 168 registers: beside a router block (256 x 64 registers) on the same SM.
template <bool Q4>
__global__ void __maxnreg__(168) dec_stream_kernel(StreamArgs a) {
  constexpr int kSpw = Q4 ? 2 : 1;  // ring slots per slot warp (items in flight per warp)
  extern __shared__ __align__(128) uint8_t ssm[];
  __shared__ int s_ids[kTopK];
  __shared__ float s_w[kTopK];
  __shared__ float s_part[kCbWarps * 4];
  __shared__ int s_fail;
  __shared__ int s_issued;  // gate/up items whose copies the slot warps have issued
  __shared__ int s_next;    // next gate/up item to hand out (items 0..7: one per slot warp)
  const int d = a.D.d, f = a.D.f, fs = a.D.fs, hdim = a.D.hdim, nch = d / 8;
  const int G = gridDim.x, b = blockIdx.x;
  const StLayout Ly = st_layout<Q4>(a.D, G);
  const uint32_t slot_bytes = Ly.slot;
  const uint32_t row_bytes = Q4 ? (uint32_t)d / 2 : (uint32_t)d * 2;  // codes / bf16 of a row
  const uint32_t grp_bytes = (uint32_t)d / 32;                        // a 4-bit row's scales
  uint8_t* ring = ssm;
  uint8_t* rows = ssm + Ly.rows;
  float* hs = reinterpret_cast<float*>(ssm + Ly.hp);
  uint64_t* full = reinterpret_cast<uint64_t*>(ssm + Ly.bars);
  uint64_t* sel_ready = full + kStSlots * kSpw;  // s_ids holds this forward's selection
  uint64_t* dbar = sel_ready + 1;         // the down rows have landed
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = (int)((long long)b * d / G), nn = (int)((long long)(b + 1) * d / G) - n0;
  // bytes per down row: bf16 rows, or codes (then scales and biases in their own regions)
  const uint32_t rb = Q4 ? (uint32_t)f / 2 : (uint32_t)f * 2;
  const uint32_t srb = Q4 ? (uint32_t)fs / 2 : (uint32_t)fs * 2;
  // this block's gate/up items: the shared expert's features b, b + G, ..., then the routed
  // features r = j f + c (j: rank of the expert in ascending id) b, b + G, ...: at any moment
  // the blocks together request consecutive rows, a few sequential sweeps for DRAM
  const int ns = fs > b ? (fs - b + G - 1) / G : 0;
  const int nr = kTopK * f;
  const int nitems = ns + (nr > b ? (nr - b + G - 1) / G : 0);
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStSlots * kSpw; ++i) mbar_init(&full[i], 1);
    mbar_init(sel_ready, 1);
    mbar_init(dbar, 1);
    s_fail = 0;
    s_issued = 0;
    s_next = kStSlots * kSpw;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_trigger();  // the next layer's router may request its rows (it waits for this launch)
  const uint64_t pol = policy_evict_first();  // every weight row is read once

  // down rows of expert rank j (j = 8: the shared expert) into shared memory, completing on dbar
  auto copy_down = [&](int j, int e) {
    if (!Q4) {
      const __nv_bfloat16* src = j < 8 ? a.W.w_down + ((size_t)e * d + n0) * f
                                       : a.W.ws_down + (size_t)n0 * fs;
      bulk_load(rows + (j < 8 ? j * nn * rb : 8 * nn * rb), src, nn * (j < 8 ? rb : srb), dbar,
                pol);
    } else {
      const Q4Matrix& m = j < 8 ? a.Q.down : a.Q.s_down;
      const int K = j < 8 ? f : fs;
      const size_t r0 = j < 8 ? (size_t)e * d + n0 : (size_t)n0;
      const uint32_t coff = j < 8 ? j * nn * (f / 2) : 8 * nn * (f / 2);
      const uint32_t goff = j < 8 ? j * nn * (f / 32) : 8 * nn * (f / 32);
      bulk_load(rows + coff, m.codes + r0 * (K / 2), nn * (K / 2), dbar, pol);
      bulk_load(ssm + Ly.sc + goff, m.scales + r0 * (K / 64), nn * (K / 32), dbar, pol);
      bulk_load(ssm + Ly.bi + goff, m.biases + r0 * (K / 64), nn * (K / 32), dbar, pol);
    }
  };

  if (warp == 0) {
    // ---- selection and the down rows
    if (lane == 0) {
      const uint32_t down_bytes =
          Q4 ? (uint32_t)nn * (8 * f + fs) * 9 / 16 : (uint32_t)nn * (8 * rb + srb);
      mbar_arrive_expect_tx(dbar, down_bytes);
      copy_down(8, 0);
    }
    pdl_wait();  // the router's logits (and x) are final
    named_arrive(2, kStThreads);  // releases the slot warps (parked on the same barrier)
    select_top8(a.dw.logits, lane, s_ids, s_w);
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      mbar_arrive(sel_ready);
    }
    // the routed down rows once the slot warps have issued all but their last items: HBM then
    // serves the gate/up rows first (the grid barrier waits for those) and the down rows during
    // the last items and the barrier (the combine after it waits for these)
    if (lane == 0) {
      const int want = nitems - kDownLead;
      const uint64_t t0 = global_timer_ns();
      while (*reinterpret_cast<volatile int*>(&s_issued) < want &&
             global_timer_ns() - t0 < kWaitLimitNs)
        __nanosleep(256);
    }
    __syncwarp();
    if (lane < kTopK) copy_down(lane, s_ids[lane]);
    if (b == 0 && lane < kTopK) {
      a.topk_idx[lane] = s_ids[lane];
      a.topk_w[lane] = s_w[lane];
    }
  } else {
    // ---- slot warp w (warp - 1) owns slots w * kSpw .. w * kSpw + kSpw - 1 (kSpw items in
    // flight per warp) and takes the block's next item whenever one of its slots is free
    const int w = warp - 1;
    // the expert row of item k (a routed item needs the selection): feature row index in
    // matrix gate/up of expert e (e < 0: the shared expert)
    auto item_row = [&](int k, int& e, size_t& r) {
      if (k < ns) {
        e = -1;
        r = (size_t)(b + k * G);
      } else {
        const int rr = b + (k - ns) * G, j = rr / f;
        e = s_ids[j];
        r = (size_t)e * f + (rr - j * f);
      }
    };
    auto issue = [&](int k, int sl_i) {  // lane 0: item k into slot sl_i
      int e;
      size_t r;
      item_row(k, e, r);
      uint8_t* sl = ring + sl_i * slot_bytes;
      uint64_t* fb = &full[sl_i];
      mbar_arrive_expect_tx(fb, slot_bytes);
      if (!Q4) {
        const __nv_bfloat16* g = (e < 0 ? a.W.ws_gate : a.W.w_gate) + r * d;
        const __nv_bfloat16* u = (e < 0 ? a.W.ws_up : a.W.w_up) + r * d;
        bulk_load(sl, g, row_bytes, fb, pol);
        bulk_load(sl + row_bytes, u, row_bytes, fb, pol);
      } else {
        const Q4Matrix& mg = e < 0 ? a.Q.s_gate : a.Q.gate;
        const Q4Matrix& mu = e < 0 ? a.Q.s_up : a.Q.up;
        bulk_load(sl, mg.codes + r * (d / 2), row_bytes, fb, pol);
        bulk_load(sl + row_bytes, mu.codes + r * (d / 2), row_bytes, fb, pol);
        bulk_load(sl + 2 * row_bytes, mg.scales + r * (d / 64), grp_bytes, fb, pol);
        bulk_load(sl + 2 * row_bytes + grp_bytes, mg.biases + r * (d / 64), grp_bytes, fb, pol);
        bulk_load(sl + 2 * row_bytes + 2 * grp_bytes, mu.scales + r * (d / 64), grp_bytes, fb,
                  pol);
        bulk_load(sl + 2 * row_bytes + 3 * grp_bytes, mu.biases + r * (d / 64), grp_bytes, fb,
                  pol);
      }
      atomicAdd(&s_issued, 1);
    };
    bool sel = false;  // lane 0 has seen the selection
    auto ensure_sel = [&]() {
      if (!sel) sel = mbar_wait(sel_ready, 0, a.err);
      return sel;
    };
    // slot t of this warp starts with item w + kStSlots * t (shared features before the
    // router has finished); later items come from s_next, in index order
    int kk[kSpw], uu[kSpw];
#pragma unroll
    for (int t = 0; t < kSpw; ++t) {
      kk[t] = w + kStSlots * t;
      uu[t] = 0;
      if (lane == 0 && kk[t] < ns) issue(kk[t], w * kSpw + t);
    }
    named_sync(2, kStThreads);  // warp 0 has passed its wait: x is final
    if (!Q4) {
      const uint4* xsrc = reinterpret_cast<const uint4*>(a.x);
      uint4* xs = reinterpret_cast<uint4*>(ssm + Ly.xs);
      for (int i = threadIdx.x - 32; i < nch; i += kStThreads - 32) xs[i] = __ldcg(xsrc + i);
      named_sync(1, kStThreads - 32);
    } else {
      stage_f32_named(a.x, reinterpret_cast<float*>(ssm + Ly.xs),
                      reinterpret_cast<float*>(ssm + Ly.xsum), d, threadIdx.x - 32,
                      kStThreads - 32, 1);
    }
    bool ok = true;
#pragma unroll
    for (int t = 0; t < kSpw; ++t)
      if (lane == 0 && kk[t] >= ns && kk[t] < nitems) {
        ok = ok && ensure_sel();
        if (ok) issue(kk[t], w * kSpw + t);
      }
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) {
#pragma unroll
      for (int t = 0; t < kSpw; ++t) kk[t] = nitems;  // (the shared items' copies are drained below)
    }
    // the rows of item i requested into L2, one 128-byte line per lane and request (the warp has
    // seen the selection if i is routed); items are handed out in index order, item i is
    // requested when item i - 2 R (R = kStSlots kSpw, the items in flight in the ring) is
    // handed out, items R .. 3R - 1 here: with bf16 rows about 190 KB per SM in flight -- HBM
    // needs about 20 MB in flight over the chip to run at full rate, far more than the ring
    // holds -- and the requests come back roughly in the order the slots consume them
    constexpr int kRing = kStSlots * kSpw;
    bool selw = false;  // the whole warp has seen the selection
    auto prefetch_ahead = [&](int i) {
      if (i >= nitems) return;
      if (i >= ns && !selw) selw = __all_sync(0xffffffffu, mbar_wait(sel_ready, 0, a.err));
      if (i >= ns && !selw) return;
      int e;
      size_t r;
      item_row(i, e, r);
      if (!Q4) {
        const char* g = reinterpret_cast<const char*>((e < 0 ? a.W.ws_gate : a.W.w_gate) + r * d);
        const char* uq = reinterpret_cast<const char*>((e < 0 ? a.W.ws_up : a.W.w_up) + r * d);
        for (uint32_t o = lane * 128u; o < row_bytes; o += 32 * 128u) {
          prefetch_l2_line(g + o);
          prefetch_l2_line(uq + o);
        }
      } else {
        const Q4Matrix& mg = e < 0 ? a.Q.s_gate : a.Q.gate;
        const Q4Matrix& mu = e < 0 ? a.Q.s_up : a.Q.up;
        for (uint32_t o = lane * 128u; o < row_bytes; o += 32 * 128u) {
          prefetch_l2_line(mg.codes + r * (d / 2) + o);
          prefetch_l2_line(mu.codes + r * (d / 2) + o);
        }
        if (lane < 4) {
          const Q4Matrix& m = lane & 1 ? mu : mg;
          prefetch_l2_line((lane & 2 ? m.biases : m.scales) + r * (d / 64));
        }
      }
    };
    if (ok)
      for (int t = kSpw; t < 3 * kSpw; ++t) prefetch_ahead(w + kStSlots * t);
    bool any = true;
    while (ok && any) {
      any = false;
#pragma unroll
      for (int t = 0; t < kSpw; ++t) {
        if (!ok || kk[t] >= nitems) continue;
        any = true;
        const int si = w * kSpw + t, k = kk[t];
        if (!__all_sync(0xffffffffu, mbar_wait(&full[si], uu[t] & 1, a.err))) {
          ok = false;
          break;
        }
        const uint8_t* sl = ring + si * slot_bytes;
        float gsum, vsum;
        if (!Q4) {
          const uint4* gr = reinterpret_cast<const uint4*>(sl);
          const uint4* ur = gr + nch;
          const uint4* xs = reinterpret_cast<const uint4*>(ssm + Ly.xs);
          float g0 = 0.f, g1 = 0.f, v0 = 0.f, v1 = 0.f;
#pragma unroll 4
          for (int c = lane; c < nch; c += 32) {
            const uint4 xv = xs[c], wg = gr[c], wu = ur[c];
            const float x0 = bf16_lo(xv.x), x1 = bf16_hi(xv.x), x2 = bf16_lo(xv.y),
                        x3 = bf16_hi(xv.y);
            const float x4 = bf16_lo(xv.z), x5 = bf16_hi(xv.z), x6 = bf16_lo(xv.w),
                        x7 = bf16_hi(xv.w);
            g0 = fmaf(bf16_lo(wg.x), x0, g0);
            g1 = fmaf(bf16_hi(wg.x), x1, g1);
            v0 = fmaf(bf16_lo(wu.x), x0, v0);
            v1 = fmaf(bf16_hi(wu.x), x1, v1);
            g0 = fmaf(bf16_lo(wg.y), x2, g0);
            g1 = fmaf(bf16_hi(wg.y), x3, g1);
            v0 = fmaf(bf16_lo(wu.y), x2, v0);
            v1 = fmaf(bf16_hi(wu.y), x3, v1);
            g0 = fmaf(bf16_lo(wg.z), x4, g0);
            g1 = fmaf(bf16_hi(wg.z), x5, g1);
            v0 = fmaf(bf16_lo(wu.z), x4, v0);
            v1 = fmaf(bf16_hi(wu.z), x5, v1);
            g0 = fmaf(bf16_lo(wg.w), x6, g0);
            g1 = fmaf(bf16_hi(wg.w), x7, g1);
            v0 = fmaf(bf16_lo(wu.w), x6, v0);
            v1 = fmaf(bf16_hi(wu.w), x7, v1);
          }
          gsum = g0 + g1;
          vsum = v0 + v1;
        } else {
          // per piece of 32 inputs: scale * codes . x + bias * sum x
          const float* xf = reinterpret_cast<const float*>(ssm + Ly.xs);
          const float* xsum = reinterpret_cast<const float*>(ssm + Ly.xsum);
          const uint8_t* gs = sl + 2 * row_bytes;
          float gp[2] = {0.f, 0.f}, vp[2] = {0.f, 0.f};  // independent per piece parity
          for (int p0 = lane; p0 < d / 32; p0 += 64) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int p = p0 + 32 * h;
              if (p < d / 32) {
                const uint4 cg = *reinterpret_cast<const uint4*>(sl + (size_t)p * 16);
                const uint4 cu = *reinterpret_cast<const uint4*>(sl + row_bytes + (size_t)p * 16);
                const float xp = xsum[p];
                gp[h] += bf16_at(gs + (p / 2) * 2) * q4_dot32(cg, xf, p) +
                         bf16_at(gs + grp_bytes + (p / 2) * 2) * xp;
                vp[h] += bf16_at(gs + 2 * grp_bytes + (p / 2) * 2) * q4_dot32(cu, xf, p) +
                         bf16_at(gs + 3 * grp_bytes + (p / 2) * 2) * xp;
              }
            }
          }
          gsum = gp[0] + gp[1];
          vsum = vp[0] + vp[1];
        }
        const float g = warp_sum(gsum), v = warp_sum(vsum);
        __syncwarp();  // every lane has read the slot: refill it
        int kn = 0;
        if (lane == 0) kn = atomicAdd(&s_next, 1);
        kn = __shfl_sync(0xffffffffu, kn, 0);
        prefetch_ahead(kn + 2 * kRing);
        bool issued = true;
        if (lane == 0 && kn < nitems) {
          if (kn < ns || ensure_sel()) issue(kn, si);
          else issued = false;
        }
        if (lane == 0) {
          int hidx;
          if (k < ns) {
            hidx = 8 * hdim + b + k * G;
          } else {
            const int rr = b + (k - ns) * G, j = rr / f;
            hidx = j * hdim + (rr - j * f);
          }
          a.dw.hdec[hidx] = silu_mul(g, v);
        }
        ++uu[t];
        kk[t] = kn;
        if (!__all_sync(0xffffffffu, issued)) {
          ok = false;
          kk[t] = nitems;  // nothing in flight in this slot
          break;
        }
      }
    }
    if (!ok) {
      // after a timeout: each slot's copy, if one is in flight, gets another bounded chance to
      // land before the block can leave; the block still takes part in every barrier below
      if (lane == 0) {
#pragma unroll
        for (int t = 0; t < kSpw; ++t)
          if (kk[t] < nitems) mbar_wait(&full[w * kSpw + t], uu[t] & 1, a.err);
        s_fail = 1;
      }
    }
  }

  // ---- grid-wide: every block's h is in global memory
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(a.dw.gu_next, 1);
    const uint64_t t0 = global_timer_ns();
    while (true) {
      int v;
      asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(a.dw.gu_next) : "memory");
      if (v >= G + a.bar_extra) break;
      if (global_timer_ns() - t0 > a.limit_ns) {
        atomicExch(a.err, kDevErrTimeout);
        s_fail = 1;
        break;
      }
    }
  }
  __syncthreads();
  {
    const float4* src = reinterpret_cast<const float4*>(a.dw.hdec);
    float4* dst = reinterpret_cast<float4*>(hs);
    const int n4 = 9 * hdim / 4, per = hdim / 4;
    for (int base = threadIdx.x; base < n4; base += 8 * kStThreads) {
      float4 v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (base + i * kStThreads < n4) v[i] = __ldcg(src + base + i * kStThreads);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int q = base + i * kStThreads;
        if (q >= n4) continue;
        if (!Q4) {
          // float4 q of h (expert rank q / (hdim / 4)) goes to plane q % 2, piece (q % per) / 2
          dst[(q & 1) * (n4 / 2) + (q / per) * (per / 2) + (q % per) / 2] = v[i];
        } else {
          // each row h_j swizzled on its own (the swizzle moves float4 groups whole)
          const int j = q / per, c = (q - j * per) * 4;
          *reinterpret_cast<float4*>(hs + j * hdim + swz(c)) = v[i];
        }
      }
    }
  }
  if (warp == 0) {
    const bool landed = mbar_wait(dbar, 0, a.err);
    // after a timeout: one more bounded chance for the copies to land before the block leaves
    if (!landed) mbar_wait(dbar, 0, a.err);
    if (lane == 0 && !landed) s_fail = 1;
  }
  __syncthreads();
  if (s_fail || warp == 0) return;
  if (!Q4)
    dn_combine_rows(rows, reinterpret_cast<const float4*>(hs), nn, f, fs, hdim, s_w, s_part,
                    a.y + n0, warp - 1, threadIdx.x - 32);
  else
    dn_combine_q4(rows, ssm + Ly.sc, ssm + Ly.bi, hs, nn, f, fs, hdim, s_w, s_part, a.y + n0,
                  warp - 1, threadIdx.x - 32);
}

}  // namespace

namespace {
int g_gateup_grid = 0, g_down_grid = 0;  // blocks that are resident at once (all SMs)
}

cudaError_t prepare_decode_kernels(int hdim) {
  const int need = 9 * hdim * (int)sizeof(float);
  cudaError_t e = cudaSuccess;
  if (need > 48 * 1024) {
    e = cudaFuncSetAttribute(dec_down_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             need);
    if (e != cudaSuccess) return e;
  }
  int dev = 0, sms = 0, b1 = 0, b2 = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b1, dec_gateup_kernel, kWarps * 32,
                                                         8192 * 2)) != cudaSuccess)
    return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b2, dec_down_combine_kernel,
                                                         kWarps * 32, need)) != cudaSuccess)
    return e;
  g_gateup_grid = sms * (b1 > 0 ? b1 : 1);
  g_down_grid = sms * (b2 > 0 ? b2 : 1);
  return cudaSuccess;
}

cudaError_t launch_decode_router_shared(const __nv_bfloat16* x, const DecodeWeights& W,
                                        const Dims& D, int32_t* topk_idx, float* topk_w,
                                        int32_t* offsets, int32_t* perm, const DecodeWs& dw,
                                        int* err, cudaStream_t s, bool with_shared) {
  RouterSharedArgs a{x, W, D, topk_idx, offsets, perm, topk_w, dw, kE / kWarps, err};
  if (!with_shared)
    return launch_pdl(dec_router_shared_kernel<false>, dim3(a.router_blocks), dim3(kWarps * 32),
                      (size_t)D.d * 2, s, a);
  const int blocks = a.router_blocks + (D.fs + kWarps - 1) / kWarps;
  return launch_pdl(dec_router_shared_kernel<true>, dim3(blocks), dim3(kWarps * 32),
                    (size_t)D.d * 2, s, a);
}

cudaError_t launch_decode_gateup(const __nv_bfloat16* x, const DecodeWeights& W, const Dims& D,
                                 int32_t* topk_idx, float* topk_w, const DecodeWs& dw,
                                 cudaStream_t s) {
  GateUpArgs a{x, W, D, topk_idx, topk_w, dw};
  const int grid = std::min(g_gateup_grid, (D.fs + kTopK * D.f) / kWarps);
  return launch_pdl(dec_gateup_kernel, dim3(grid), dim3(kWarps * 32), (size_t)D.d * 2, s, a);
}

cudaError_t launch_decode_down_combine(const DecodeWeights& W, const Dims& D, const DecodeWs& dw,
                                       __nv_bfloat16* y, cudaStream_t s) {
  DownArgs a{W, D, dw, y};
  const int grid = std::min(g_down_grid, (D.d + kWarps - 1) / kWarps);
  return launch_pdl(dec_down_combine_kernel, dim3(grid), dim3(kWarps * 32),
                    (size_t)9 * D.hdim * sizeof(float), s, a);
}

// ---- streamed batch-1 decode

namespace {
int stream_grid(const Dims& D, int sms) { return D.d < sms ? D.d : sms; }
}  // namespace

bool decode_stream_fits(const Dims& D, int sms, bool q4) {
  const int G = stream_grid(D, sms);
  if (D.d > kStreamMaxD || (D.d + G - 1) / G > kStMaxOut) return false;
  // 4-bit: a row's scales (K / 64 bf16) must fill whole 16-byte pieces for the bulk copies
  if (q4) return D.d % 512 == 0 && D.f % 512 == 0 && D.fs % 512 == 0 &&
                 st_layout<true>(D, G).total <= (uint32_t)kStreamMaxSmem;
  return st_layout<false>(D, G).total <= (uint32_t)kStreamMaxSmem;
}

cudaError_t prepare_decode_stream_kernels() {
  cudaError_t e;
  // an SM's split between L1 and shared memory is set when a block starts on an idle SM: both
  // launches of a layer ask for the largest shared memory, so that the next layer's router
  // block fits beside a streaming block
  const void* ks[3] = {reinterpret_cast<const void*>(dec_stream_kernel<false>),
                       reinterpret_cast<const void*>(dec_stream_kernel<true>),
                       reinterpret_cast<const void*>(dec_router_shared_kernel<false>)};
  for (int i = 0; i < 3; ++i) {
    if (i < 2 && (e = cudaFuncSetAttribute(ks[i], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kStreamMaxSmem)) != cudaSuccess)
      return e;
    if ((e = cudaFuncSetAttribute(ks[i], cudaFuncAttributePreferredSharedMemoryCarveout,
                                  cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
      return e;
  }
  return cudaSuccess;
}

cudaError_t launch_decode_stream(const __nv_bfloat16* x, const DecodeWeights& W, const Dims& D,
                                 int32_t* topk_idx, float* topk_w, const DecodeWs& dw,
                                 __nv_bfloat16* y, int* err, int sms, cudaStream_t s,
                                 bool expire, const Q4Weights* q4) {
  // expire: one arrival more than the launch has, 1 ms limit (the barrier's timeout path)
  StreamArgs a{x, W, q4 ? *q4 : Q4Weights{}, D, topk_idx, topk_w, dw, y, err, expire ? 1 : 0,
               expire ? 1000000ull : kWaitLimitNs};
  const int G = stream_grid(D, sms);
  if (q4)
    return launch_pdl(dec_stream_kernel<true>, dim3(G), dim3(kStThreads),
                      st_layout<true>(D, G).total, s, a);
  return launch_pdl(dec_stream_kernel<false>, dim3(G), dim3(kStThreads),
                    st_layout<false>(D, G).total, s, a);
}

// ---- small batches

bool decode_batch_fits(const Dims& D, int T) {
  return T >= 2 && T <= kGemvMaxTokens && T * D.hdim <= kBatchMaxTHdim &&
         T * D.d <= kBatchMaxTD;
}

namespace {
// Calls f(std::integral_constant<int, T>{}) for T = 1..kGemvMaxTokens (the token count of a
// small batch as a compile-time constant); other T: invalid value.
template <class F>
cudaError_t batch_dispatch(int T, F&& f) {
  switch (T) {
    case 1: return f(std::integral_constant<int, 1>{});
    case 2: return f(std::integral_constant<int, 2>{});
    case 3: return f(std::integral_constant<int, 3>{});
    case 4: return f(std::integral_constant<int, 4>{});
    case 5: return f(std::integral_constant<int, 5>{});
    case 6: return f(std::integral_constant<int, 6>{});
    case 7: return f(std::integral_constant<int, 7>{});
    case 8: return f(std::integral_constant<int, 8>{});
    default: return cudaErrorInvalidValue;
  }
}
static_assert(kGemvMaxTokens == 8, "batch_dispatch covers 1..kGemvMaxTokens");
}  // namespace

cudaError_t prepare_decode_batch_kernels() {
  cudaError_t e;
  const int xs = kBatchMaxTD * 2, hs = kBatchMaxTHdim * 9 * 4;
  for (int T = 1; T <= kGemvMaxTokens; ++T) {
    e = batch_dispatch(T, [&](auto tt) {
      constexpr int TT = decltype(tt)::value;
      cudaError_t r = cudaFuncSetAttribute(dec_batch_router_shared_kernel<TT>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, xs);
      if (r != cudaSuccess) return r;
      r = cudaFuncSetAttribute(dec_batch_gateup_kernel<TT>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, xs);
      if (r != cudaSuccess) return r;
      return cudaFuncSetAttribute(dec_batch_down_combine_kernel<TT>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, hs);
    });
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_decode_batch_router_shared(const __nv_bfloat16* x, const DecodeWeights& W,
                                              const Dims& D, int T, int32_t* topk_idx,
                                              float* topk_w, int32_t* offsets, int32_t* perm,
                                              const DecodeWs& dw, cudaStream_t s,
                                              bool with_shared, const RouteWs* plan) {
  BatchRouterArgs a{x, W, D, T, topk_idx, offsets, perm, topk_w, dw, kE / kWarps, plan != nullptr,
                    plan_args(T, D), plan ? *plan : RouteWs{}};
  const int blocks = a.router_blocks + (with_shared ? (D.fs + kWarps - 1) / kWarps : 0);
  return batch_dispatch(T, [&](auto tt) {
    return launch_pdl(dec_batch_router_shared_kernel<decltype(tt)::value>, dim3(blocks),
                      dim3(kWarps * 32), (size_t)T * D.d * 2, s, a);
  });
}

cudaError_t launch_decode_batch_gateup(const __nv_bfloat16* x, const DecodeWeights& W,
                                       const Dims& D, int T, int32_t* topk_idx, float* topk_w,
                                       const DecodeWs& dw, int sms, cudaStream_t s) {
  BatchGateUpArgs a{x, W, D, T, topk_idx, topk_w, dw};
  return batch_dispatch(T, [&](auto tt) {
    return launch_pdl(dec_batch_gateup_kernel<decltype(tt)::value>, dim3(2 * sms),
                      dim3(kWarps * 32), (size_t)T * D.d * 2, s, a);
  });
}

cudaError_t launch_decode_batch_down_combine(const DecodeWeights& W, const Dims& D, int T,
                                             const DecodeWs& dw, __nv_bfloat16* y, int sms,
                                             cudaStream_t s) {
  BatchDownArgs a{W, D, T, dw, y};
  const int grid = std::min(2 * sms, (D.d + kWarps - 1) / kWarps);
  return batch_dispatch(T, [&](auto tt) {
    return launch_pdl(dec_batch_down_combine_kernel<decltype(tt)::value>, dim3(grid),
                      dim3(kWarps * 32), (size_t)T * 9 * D.hdim * sizeof(float), s, a);
  });
}

}  // namespace moe
