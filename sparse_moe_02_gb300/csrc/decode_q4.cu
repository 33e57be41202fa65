// Batch-1 decode with 4-bit group-affine expert weights ("Optimizing on-device inference for
// Apple Silicon", § "Dequantize weights during matrix multiplication": 4-bit weights in groups
// of 64 with a scale and a bias, dequantized inside the matrix kernel; § "Optimize the
// one-row weight path"; § "Reduce intermediate and state traffic").
//
// Same three launches as the bf16 decode path (router + shared gate/up; the 8 selected
// experts' gate/up with SwiGLU; down rows weighted and combined in fixed order), but every
// expert row is 4-bit: one 16-byte load carries 32 codes, i.e. half a group, and the piece's
// contribution is scale * sum_i q_i v_i + bias * sum_i v_i over its 32 inputs v (the sums of v
// per 32 inputs are formed once per block).  The router stays bf16.  Codes are turned into
// floats exactly: 0x4B000000 | q is the float 2^23 + q.
#include <algorithm>

#include "layer.cuh"
#include "ptx.cuh"
#include "select.cuh"
#include "q4.cuh"

namespace moe {
namespace {

constexpr int kQWarps = 8;  // warps per block in every 4-bit decode kernel
constexpr int kQB = 2;      // 16-byte code pieces per lane and row held in flight

__device__ __forceinline__ float warp_sum_q(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Up to kQB pieces per lane of one 4-bit row of np pieces: piece p = p0 + lane + 32 i, with
// its group's scale and bias.
struct Q4Frag {
  uint4 c[kQB];
  float s[kQB], b[kQB];
};

__device__ __forceinline__ void q4_load(Q4Frag& r, const Q4Row& row, int np, int lane, int p0) {
#pragma unroll
  for (int i = 0; i < kQB; ++i) {
    const int p = p0 + lane + 32 * i;
    if (p < np) {
      r.c[i] = ld_stream_u4(row.codes + (size_t)p * 16);
      r.s[i] = ld_bf16(row.scales + p / 2);
      r.b[i] = ld_bf16(row.biases + p / 2);
    }
  }
}

// Lane-partial of row . v for the pieces in r (v and its per-32 sums vs in shared memory).
__device__ __forceinline__ float q4_dot(const Q4Frag& r, const float* v, const float* vs, int np,
                                        int lane, int p0) {
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < kQB; ++i) {
    const int p = p0 + lane + 32 * i;
    if (p < np) acc += r.s[i] * q4_dot32(r.c[i], v, p) + r.b[i] * vs[p];
  }
  return acc;
}

// Lane-partial of row . v over the whole row; the first kQB*32 pieces already in r.
__device__ __forceinline__ float q4_dot_rest(Q4Frag& r, const Q4Row& row, const float* v,
                                             const float* vs, int np, int lane) {
  float acc = q4_dot(r, v, vs, np, lane, 0);
  for (int p0 = kQB * 32; p0 < np; p0 += kQB * 32) {
    q4_load(r, row, np, lane, p0);
    acc += q4_dot(r, v, vs, np, lane, p0);
  }
  return acc;
}

// Stages v (n bf16 values, n a multiple of 32) as fp32, swizzled, in vf[n] and the sums of
// each 32 (ascending) in vs[n / 32]; every thread of the block calls this (it holds barriers).
__device__ __forceinline__ void stage_f32(const __nv_bfloat16* src, float* vf, float* vs, int n) {
  // 8 elements per 16-byte load, up to four loads of a thread in flight before its stores (one
  // round trip per batch); the swizzle moves groups of 4 whole, so each half of a load is one
  // float4 store
  const uint4* s16 = reinterpret_cast<const uint4*>(src);
  const int n8 = n / 8;
  for (int base = threadIdx.x; base < n8; base += 4 * blockDim.x) {
    uint4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (base + i * (int)blockDim.x < n8) v[i] = s16[base + i * blockDim.x];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int m = base + i * (int)blockDim.x;
      if (m < n8) {
        *reinterpret_cast<float4*>(vf + swz(8 * m)) =
            make_float4(bf16_lo(v[i].x), bf16_hi(v[i].x), bf16_lo(v[i].y), bf16_hi(v[i].y));
        *reinterpret_cast<float4*>(vf + swz(8 * m + 4)) =
            make_float4(bf16_lo(v[i].z), bf16_hi(v[i].z), bf16_lo(v[i].w), bf16_hi(v[i].w));
      }
    }
  }
  __syncthreads();
  // a piece's 32 values are its 32 slots in some order: summed in slot order
  for (int p = threadIdx.x; p < n / 32; p += blockDim.x) {
    const float4* q = reinterpret_cast<const float4*>(vf + 32 * p);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 t = q[i];
      s += t.x;
      s += t.y;
      s += t.z;
      s += t.w;
    }
    vs[p] = s;
  }
  __syncthreads();
}

struct Q4GateUpArgs {
  const __nv_bfloat16* x;
  Q4Weights W;
  Dims D;
  int32_t* topk_idx;  // written by block 0 (the selection behind this forward)
  float* topk_w;
  DecodeWs dw;
};

// Items, one warp per item over a resident grid: first the shared expert's features c < fs,
// then the selected experts' (j, c): h[j][c] = silu(gate . x) * (up . x) from the 4-bit gate
// and up rows.  A warp whose first item is a shared feature requests its rows before waiting
// on the router kernel.  Warp 0 of every block selects the top 8 from the router logits first.
__global__ void __launch_bounds__(kQWarps * 32, 2) dec_q4_gateup_kernel(Q4GateUpArgs a) {
  extern __shared__ float qsm[];
  float* xf = qsm;
  float* xs = qsm + a.D.d;
  __shared__ int s_ids[kTopK];
  __shared__ float s_w[kTopK];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.D.d, f = a.D.f, fs = a.D.fs, np = d / 32;
  const int total = fs + kTopK * f;
  const int nwarps = gridDim.x * kQWarps;
  int it = blockIdx.x * kQWarps + warp;
  Q4Frag g, u;
  if (it < fs) {
    q4_load(g, a.W.s_gate.row(it, d), np, lane, 0);
    q4_load(u, a.W.s_up.row(it, d), np, lane, 0);
  }
  pdl_wait();     // the router logits come from the previous kernel
  pdl_trigger();  // the down kernel may start selecting and streaming its rows now
  if (warp == 0) select_top8(a.dw.logits, lane, s_ids, s_w);
  stage_f32(a.x, xf, xs, d);
  if (blockIdx.x == 0 && threadIdx.x < kTopK) {
    a.topk_idx[threadIdx.x] = s_ids[threadIdx.x];
    a.topk_w[threadIdx.x] = s_w[threadIdx.x];
  }
  for (bool first = true; it < total; it += nwarps, first = false) {
    Q4Row rg, ru;
    size_t slot;
    if (it < fs) {
      rg = a.W.s_gate.row(it, d);
      ru = a.W.s_up.row(it, d);
      slot = (size_t)8 * a.D.hdim + it;
    } else {
      const int j = (it - fs) / f, c = (it - fs) % f;
      const size_t r = (size_t)s_ids[j] * f + c;
      rg = a.W.gate.row(r, d);
      ru = a.W.up.row(r, d);
      slot = (size_t)j * a.D.hdim + c;
    }
    if (!(first && it < fs)) {  // the first shared item's pieces are already in registers
      q4_load(g, rg, np, lane, 0);
      q4_load(u, ru, np, lane, 0);
    }
    const float gv = warp_sum_q(q4_dot_rest(g, rg, xf, xs, np, lane));
    const float uv = warp_sum_q(q4_dot_rest(u, ru, xf, xs, np, lane));
    if (lane == 0) a.dw.hdec[slot] = silu_mul(gv, uv);
  }
}

struct Q4DownArgs {
  Q4Weights W;
  Dims D;
  DecodeWs dw;
  __nv_bfloat16* y;
};

constexpr int kQDPre = 6;  // pieces per lane of one output's nine down rows held in flight

// One warp per output n over a resident grid.  The nine 4-bit down rows of n (experts
// j = 0..7 in ascending id, then the shared expert) are taken as one run of pieces, piece P of
// routed row j = P / (f/32) or of the shared row past 8 f/32; lane l takes P = l, l+32, ...
// and sums w_j (scale * codes . h_j + bias * sum h_j) over its pieces in that order; one warp
// reduction gives y[n].  The top 8 is selected again from the router logits (final: the router
// kernel completed before the gate/up kernel let this one start), so the first output's rows
// are requested before waiting for h.
__global__ void __launch_bounds__(kQWarps * 32, 2) dec_q4_down_combine_kernel(Q4DownArgs a) {
  extern __shared__ float qsm[];  // h [9][hdim] fp32, then its sums per 32 [9][hdim / 32]
  const int d = a.D.d, f = a.D.f, fs = a.D.fs, hdim = a.D.hdim;
  float* hf = qsm;
  float* hsum = qsm + 9 * hdim;
  __shared__ int s_ids[kTopK];
  __shared__ float s_w[kTopK];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) select_top8(a.dw.logits, lane, s_ids, s_w);
  __syncthreads();
  const int npr = f / 32, nps = fs / 32, npt = 8 * npr + nps;
  // the row and piece of run position P: routed row j = P / npr or the shared row (j = 8)
  auto split = [&](int P, int& j, int& p) {
    j = P < 8 * npr ? P / npr : 8;
    p = P - j * npr;
  };
  auto row_of = [&](int j, int nn) {
    return j < 8 ? a.W.down.row((size_t)s_ids[j] * d + nn, f) : a.W.s_down.row((size_t)nn, fs);
  };
  // the first kQDPre run positions of this lane are the same for every output: their rows
  // and pieces are worked out once
  int pj[kQDPre], pp[kQDPre];
#pragma unroll
  for (int i = 0; i < kQDPre; ++i) split(lane + 32 * i, pj[i], pp[i]);
  uint4 pc[kQDPre];
  float ps[kQDPre], pb[kQDPre];
  auto load = [&](int P0, int nn) {
#pragma unroll
    for (int i = 0; i < kQDPre; ++i) {
      const int P = P0 + lane + 32 * i;
      if (P < npt) {
        int j = pj[i], p = pp[i];
        if (P0) split(P, j, p);
        const Q4Row r = row_of(j, nn);
        pc[i] = ld_stream_u4(r.codes + (size_t)p * 16);
        ps[i] = ld_bf16(r.scales + p / 2);
        pb[i] = ld_bf16(r.biases + p / 2);
      }
    }
  };
  const int nwarps = gridDim.x * kQWarps;
  int n = blockIdx.x * kQWarps + warp;
  if (n < d) load(0, n);
  pdl_wait();  // h comes from the gate/up kernel
  pdl_trigger();
  // each row h_j swizzled on its own (pieces counted from the row's start), in float4 groups,
  // which the swizzle moves whole: eight 16-byte loads of a thread in flight before its stores
  // (one round trip per batch), then the sums per 32 from shared memory
  {
    const float4* src = reinterpret_cast<const float4*>(a.dw.hdec);
    const int r4 = hdim / 4, n4 = 9 * r4;
    for (int base = threadIdx.x; base < n4; base += 8 * blockDim.x) {
      float4 v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (base + i * (int)blockDim.x < n4) v[i] = __ldcg(src + base + i * blockDim.x);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int q = base + i * (int)blockDim.x;
        if (q < n4) {
          const int j = q / r4, c = (q - j * r4) * 4;
          *reinterpret_cast<float4*>(hf + j * hdim + swz(c)) = v[i];
        }
      }
    }
  }
  __syncthreads();
  // a piece's 32 values are its 32 slots in some order: summed in slot order
  for (int q = threadIdx.x; q < 9 * (hdim / 32); q += blockDim.x) {
    const float4* t4 = reinterpret_cast<const float4*>(hf + 32 * q);
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 t = t4[i];
      sum += t.x;
      sum += t.y;
      sum += t.z;
      sum += t.w;
    }
    hsum[q] = sum;
  }
  __syncthreads();
  const float wj[9] = {s_w[0], s_w[1], s_w[2], s_w[3], s_w[4], s_w[5], s_w[6], s_w[7], 1.0f};
  for (; n < d; n += nwarps) {
    float yv = 0.f;
    for (int P0 = 0; P0 < npt; P0 += 32 * kQDPre) {
      if (P0) load(P0, n);
#pragma unroll
      for (int i = 0; i < kQDPre; ++i) {
        const int P = P0 + lane + 32 * i;
        if (P < npt) {
          int j = pj[i], p = pp[i];
          if (P0) split(P, j, p);
          const float part = ps[i] * q4_dot32(pc[i], hf + (size_t)j * hdim, p) +
                             pb[i] * hsum[j * (hdim / 32) + p];
          float w = wj[0];
#pragma unroll
          for (int q = 1; q < 9; ++q) w = j == q ? wj[q] : w;
          yv = fmaf(w, part, yv);
        }
      }
    }
    yv = warp_sum_q(yv);
    if (lane == 0) a.y[n] = __float2bfloat16_rn(yv);
    if (n + nwarps < d) load(0, n + nwarps);
  }
}

}  // namespace

cudaError_t prepare_decode_q4_kernels() {
  // dynamic shared memory at the largest supported shape (d = 8192, hdim = 2048)
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(dec_q4_gateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                8192 * 4 + 256 * 4)) != cudaSuccess)
    return e;
  return cudaFuncSetAttribute(dec_q4_down_combine_kernel,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              9 * 2048 * 4 + 9 * 64 * 4);
}

cudaError_t launch_decode_q4_gateup(const __nv_bfloat16* x, const Q4Weights& W, const Dims& D,
                                    int32_t* topk_idx, float* topk_w, const DecodeWs& dw,
                                    int sms, cudaStream_t s) {
  Q4GateUpArgs a{x, W, D, topk_idx, topk_w, dw};
  const int grid = std::min(2 * sms, (D.fs + kTopK * D.f) / kQWarps);
  return launch_pdl(dec_q4_gateup_kernel, dim3(grid), dim3(kQWarps * 32),
                    (size_t)D.d * 4 + (size_t)D.d / 32 * 4, s, a);
}

cudaError_t launch_decode_q4_down_combine(const Q4Weights& W, const Dims& D, const DecodeWs& dw,
                                          __nv_bfloat16* y, int sms, cudaStream_t s) {
  Q4DownArgs a{W, D, dw, y};
  const int grid = std::min(2 * sms, (D.d + kQWarps - 1) / kQWarps);
  return launch_pdl(dec_q4_down_combine_kernel, dim3(grid), dim3(kQWarps * 32),
                    (size_t)9 * D.hdim * 4 + (size_t)9 * (D.hdim / 32) * 4, s, a);
}

}  // namespace moe
