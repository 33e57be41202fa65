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
#include "layer.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kWarps = 8;  // warps per block in every decode kernel

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

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Partial dot product of one bf16 row (nch 16-byte chunks) with x in shared memory.
__device__ __forceinline__ float row_dot_partial(const __nv_bfloat16* row, const uint4* xs,
                                                 int nch, int lane) {
  float acc = 0.f;
#pragma unroll 4
  for (int c = lane; c < nch; c += 32) acc += dot8(ld_stream_u4(row + (size_t)c * 8), xs[c]);
  return acc;
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

__global__ void __launch_bounds__(kWarps * 32) dec_router_shared_kernel(RouterSharedArgs a) {
  extern __shared__ uint4 xs[];
  __shared__ int s_last;
  __shared__ int s_ids[kTopK];
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.D.d, nch = d / 8;
  stage_x(a.x, xs, d);

  if ((int)blockIdx.x >= a.router_blocks) {
    // shared expert: h_s[c] = silu(gate_c . x) * (up_c . x), one feature per warp
    const int c = ((int)blockIdx.x - a.router_blocks) * kWarps + warp;
    if (c < a.D.fs) {
      const float g = warp_sum(row_dot_partial(a.W.ws_gate + (size_t)c * d, xs, nch, lane));
      const float u = warp_sum(row_dot_partial(a.W.ws_up + (size_t)c * d, xs, nch, lane));
      if (lane == 0) a.dw.hdec[(size_t)8 * a.D.hdim + c] = silu_mul(g, u);
    }
    pdl_trigger();
    return;
  }

  // router rows: logits[e] = w_r[e] . x (+ bias[e])
  for (int e = blockIdx.x * kWarps + warp; e < kE; e += a.router_blocks * kWarps) {
    float l = warp_sum(row_dot_partial(a.W.w_r + (size_t)e * d, xs, nch, lane));
    if (lane == 0) a.dw.logits[e] = l + (a.W.bias ? a.W.bias[e] : 0.f);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(a.dw.counter, 1) == a.router_blocks - 1;
  }
  __syncthreads();
  if (!s_last) {
    pdl_trigger();
    return;
  }
  // last router block: top-8 of the 256 logits by 8 rounds of warp arg-max (ties: lower id)
  __threadfence();
  if (warp == 0) {
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __ldcg(a.dw.logits + lane + 32 * i);
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
    // ascending expert id, then softmax over the kept logits
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
      a.topk_idx[lane] = myi;
      a.topk_w[lane] = myw / s;
      s_ids[lane] = myi;
      if (a.perm) a.perm[lane] = lane;  // one token: slot j holds assignment (0, j)
    }
    if (lane == 0) *a.dw.counter = 0;  // ready for the next launch on the stream
  }
  __syncthreads();
  if (a.offsets) {
    for (int e = threadIdx.x; e <= kE; e += blockDim.x) {
      int n = 0;
#pragma unroll
      for (int j = 0; j < kTopK; ++j) n += s_ids[j] < e;
      a.offsets[e] = n;
    }
  }
  pdl_trigger();
}

struct GateUpArgs {
  const __nv_bfloat16* x;
  DecodeWeights W;
  Dims D;
  const int32_t* topk_idx;
  DecodeWs dw;
};

// One warp per (selected expert j, feature c): h[j][c] = silu(gate . x) * (up . x).
__global__ void __launch_bounds__(kWarps * 32) dec_gateup_kernel(GateUpArgs a) {
  extern __shared__ uint4 xs[];
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.D.d, f = a.D.f, nch = d / 8;
  stage_x(a.x, xs, d);
  const int gw = blockIdx.x * kWarps + warp;
  const int j = gw / f, c = gw % f;
  if (j < kTopK) {
    const size_t row = ((size_t)a.topk_idx[j] * f + c) * d;
    const float g = warp_sum(row_dot_partial(a.W.w_gate + row, xs, nch, lane));
    const float u = warp_sum(row_dot_partial(a.W.w_up + row, xs, nch, lane));
    if (lane == 0) a.dw.hdec[(size_t)j * a.D.hdim + c] = silu_mul(g, u);
  }
  pdl_trigger();
}

struct DownArgs {
  DecodeWeights W;
  Dims D;
  const int32_t* topk_idx;
  const float* topk_w;
  DecodeWs dw;
  __nv_bfloat16* y;
};

// One warp per output n: o_j = down_{e_j}[n] . h_j for the 8 experts and the shared expert;
// y[n] = bf16(sum_j w_j o_j (ascending expert id) + o_shared), accumulated in fp32.
__global__ void __launch_bounds__(kWarps * 32) dec_down_combine_kernel(DownArgs a) {
  extern __shared__ float hs[];  // [9][hdim]
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.D.d, f = a.D.f, fs = a.D.fs, hdim = a.D.hdim;
  for (int i = threadIdx.x; i < 9 * hdim; i += blockDim.x) hs[i] = a.dw.hdec[i];
  __syncthreads();
  const int n = blockIdx.x * kWarps + warp;
  if (n < d) {
    float p[9];
#pragma unroll
    for (int j = 0; j < 9; ++j) {
      const int len = j < 8 ? f : fs;
      const __nv_bfloat16* row = j < 8 ? a.W.w_down + ((size_t)a.topk_idx[j] * d + n) * f
                                       : a.W.ws_down + (size_t)n * fs;
      const float* hj = hs + (size_t)j * hdim;
      float acc = 0.f;
#pragma unroll 2
      for (int c = lane; c < len / 8; c += 32) {
        const uint4 w = ld_stream_u4(row + (size_t)c * 8);
        const float4 h0 = *reinterpret_cast<const float4*>(hj + c * 8);
        const float4 h1 = *reinterpret_cast<const float4*>(hj + c * 8 + 4);
        acc = fmaf(bf16_lo(w.x), h0.x, acc);
        acc = fmaf(bf16_hi(w.x), h0.y, acc);
        acc = fmaf(bf16_lo(w.y), h0.z, acc);
        acc = fmaf(bf16_hi(w.y), h0.w, acc);
        acc = fmaf(bf16_lo(w.z), h1.x, acc);
        acc = fmaf(bf16_hi(w.z), h1.y, acc);
        acc = fmaf(bf16_lo(w.w), h1.z, acc);
        acc = fmaf(bf16_hi(w.w), h1.w, acc);
      }
      p[j] = acc;
    }
    float y = 0.f;
#pragma unroll
    for (int j = 0; j < 9; ++j) {
      const float o = warp_sum(p[j]);
      y += (j < 8 ? a.topk_w[j] : 1.0f) * o;
    }
    if (lane == 0) a.y[n] = __float2bfloat16_rn(y);
  }
  pdl_trigger();
}

}  // namespace

cudaError_t prepare_decode_kernels(int hdim) {
  const int need = 9 * hdim * (int)sizeof(float);
  if (need <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(dec_down_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              need);
}

cudaError_t launch_decode_router_shared(const __nv_bfloat16* x, const DecodeWeights& W,
                                        const Dims& D, int32_t* topk_idx, float* topk_w,
                                        int32_t* offsets, int32_t* perm, const DecodeWs& dw,
                                        int* err, cudaStream_t s, bool with_shared) {
  RouterSharedArgs a{x, W, D, topk_idx, offsets, perm, topk_w, dw, kE / kWarps, err};
  const int blocks = a.router_blocks + (with_shared ? (D.fs + kWarps - 1) / kWarps : 0);
  return launch_pdl(dec_router_shared_kernel, dim3(blocks), dim3(kWarps * 32),
                    (size_t)D.d * 2, s, a);
}

cudaError_t launch_decode_gateup(const __nv_bfloat16* x, const DecodeWeights& W, const Dims& D,
                                 const int32_t* topk_idx, const DecodeWs& dw, cudaStream_t s) {
  GateUpArgs a{x, W, D, topk_idx, dw};
  return launch_pdl(dec_gateup_kernel, dim3(kTopK * D.f / kWarps), dim3(kWarps * 32),
                    (size_t)D.d * 2, s, a);
}

cudaError_t launch_decode_down_combine(const DecodeWeights& W, const Dims& D,
                                       const int32_t* topk_idx, const float* topk_w,
                                       const DecodeWs& dw, __nv_bfloat16* y, cudaStream_t s) {
  DownArgs a{W, D, topk_idx, topk_w, dw, y};
  return launch_pdl(dec_down_combine_kernel, dim3((D.d + kWarps - 1) / kWarps),
                    dim3(kWarps * 32), (size_t)9 * D.hdim * sizeof(float), s, a);
}

}  // namespace moe
