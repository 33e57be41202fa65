// Gated DeltaNet recurrent scan (include/gdn.h states the rule, layouts and errors).
//
// "Optimizing on-device inference for Apple Silicon", § "Keep recurrent state on chip": one
// lane group per state column, the column held in registers for the whole scan, partial sums
// exchanged between lanes by shuffles, the state written back once at the end.
//
// GB300 layout of the work: a block owns one head and 32 value columns (grid: dv/32 x H).
// Eight consumer warps hold the 32 columns, four per warp: the 8 lanes of a group own one
// column, lane r holding the 16 key rows 4(r + 8c) + e (c, e < 4) as fp32 registers.  Per token
// a lane takes its 16-row partial sums of S^T k and S^T q, three xor-shuffle rounds complete
// them over the group, and every lane updates its rows.  Four more warps stage the tokens: chunks
// of 32 tokens' k, q (one head), v (the block's 32 columns) and gates come in by cp.async three
// chunks ahead, are widened once to fp32 (with k . q per token) into one of two shared-memory
// chunk buffers, and the outputs the consumers leave in shared memory go out in 64-byte rows.
// One block barrier per chunk hands the buffers over; nothing waits on a flag, so nothing can
// hang.  The work is fp32 FMA-bound: 4 FMA-pipe operations per state element and token.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace {

constexpr int kDk = 128;
constexpr int kCols = 32;                     // value columns per block
constexpr int kCWarps = 8;                    // consumer warps, 4 columns each
constexpr int kSWarps = 4;                    // staging warps, 8 tokens of a chunk each
constexpr int kThreads = 32 * (kCWarps + kSWarps);
constexpr int kTc = 32;                       // tokens per chunk
constexpr int kRawStages = 3;                 // bf16 chunks in flight

// Shared memory, bytes.  Raw stage: k, q [kTc][256] (16-byte pieces p of token t at slot
// p ^ (t & 7)), v [kTc][64], alpha, beta [kTc].  fp32 stage: k, q [kTc][512] (4-float piece P
// of token t at slot P ^ (t & 7)), v [kTc][32], gates [kTc] x (alpha, beta, k . q, 0).  Output
// stage: [kTc][32] bf16.  The xor swizzles keep the staging warp's per-token rows and the
// consumers' per-piece reads free of bank conflicts.
constexpr int kRawK = 0;
constexpr int kRawQ = kRawK + kTc * 256;
constexpr int kRawV = kRawQ + kTc * 256;
constexpr int kRawA = kRawV + kTc * 64;
constexpr int kRawB = kRawA + kTc * 4;
constexpr int kRawBytes = kRawB + kTc * 4;
constexpr int kFK = 0;
constexpr int kFQ = kFK + kTc * 512;
constexpr int kFV = kFQ + kTc * 512;
constexpr int kFG = kFV + kTc * kCols * 4;
constexpr int kFBytes = kFG + kTc * 16;
constexpr int kOBytes = kTc * kCols * 2;
constexpr int kRawOff = 0;
constexpr int kFOff = kRawOff + kRawStages * kRawBytes;
constexpr int kOOff = kFOff + 2 * kFBytes;
constexpr int kSmemBytes = kOOff + 2 * kOBytes;
static_assert(kRawBytes % 16 == 0 && kFBytes % 16 == 0 && kOBytes % 16 == 0, "16-byte stages");

struct ScanArgs {
  const uint8_t* q;
  const uint8_t* k;
  const uint8_t* v;
  const float* alpha;
  const float* beta;
  const float* s_in;
  float* s_out;
  uint8_t* o;
  int64_t T;
  int H;
  int dv;
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}

// At most two groups of this thread still pending.
__device__ __forceinline__ void cp_async_wait2() {
  asm volatile("cp.async.wait_group 2;\n" ::: "memory");
}

// bf16 pairs of a 32-bit word -> fp32 (exact): element 2m in the low half.
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ int64_t chunk_tokens(int64_t T, int64_t cc) {
  const int64_t left = T - cc * kTc;
  return left <= 0 ? 0 : (left < kTc ? left : kTc);
}

// ---- staging warps
//
// Staging warp w (one per SM sub-partition, so that the staging work is spread evenly over the
// four schedulers) owns tokens 8w .. 8w + 7 of every chunk: it copies their inputs, widens them
// and writes their outputs.  Lane l of it works on token 8w + l / 4, quarter l % 4 of the row.

// cp.async of this warp's tokens of chunk cc into raw stage rs (one commit group, empty past
// the end of the prompt).
__device__ __forceinline__ void stage_issue(const ScanArgs& a, uint8_t* rs, int64_t cc, int h,
                                            int c0, int sw_warp, int lane) {
  const int64_t n = chunk_tokens(a.T, cc);
  const int64_t t0 = cc * kTc;
#pragma unroll
  for (int it = 0; it < 4; ++it) {  // two tokens' 256-byte k and q rows per instruction
    const int tl = 8 * sw_warp + 2 * it + (lane >> 4), p = lane & 15;
    if (tl < n) {
      const int64_t row = ((t0 + tl) * a.H + h) * (kDk * 2);
      const int slot = (p ^ (tl & 7)) * 16;
      cp_async16(rs + kRawK + tl * 256 + slot, a.k + row + p * 16);
      cp_async16(rs + kRawQ + tl * 256 + slot, a.q + row + p * 16);
    }
  }
  {  // eight tokens' 64-byte v slices
    const int tl = 8 * sw_warp + (lane >> 2), pc = lane & 3;
    if (tl < n)
      cp_async16(rs + kRawV + tl * 64 + pc * 16,
                 a.v + ((t0 + tl) * a.H + h) * (int64_t)a.dv * 2 + (int64_t)c0 * 2 + pc * 16);
  }
  if (lane < 8 && 8 * sw_warp + lane < n) {
    const int tl = 8 * sw_warp + lane;
    cp_async4(rs + kRawA + tl * 4, a.alpha + (t0 + tl) * a.H + h);
    cp_async4(rs + kRawB + tl * 4, a.beta + (t0 + tl) * a.H + h);
  }
  cp_async_commit();
}

// Widens this warp's tokens of chunk cc from raw stage rs into fp32 stage fs, with k . q per
// token: each lane sums its quarter (32 products, ascending index), then the four quarters are
// added by two xor shuffles (the same tree in every lane).
__device__ __forceinline__ void stage_convert(const ScanArgs& a, const uint8_t* rs, uint8_t* fs,
                                              int64_t cc, int sw_warp, int lane) {
  const int tl = 8 * sw_warp + (lane >> 2), qd = lane & 3;
  const bool live = tl < chunk_tokens(a.T, cc);
  const int sw = tl & 7;
  float qk = 0.f;
  if (live) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int p = 4 * qd + i;
      const uint4 rk = *reinterpret_cast<const uint4*>(rs + kRawK + tl * 256 + (p ^ sw) * 16);
      const uint4 rq = *reinterpret_cast<const uint4*>(rs + kRawQ + tl * 256 + (p ^ sw) * 16);
      const float4 k0 = make_float4(bf_lo(rk.x), bf_hi(rk.x), bf_lo(rk.y), bf_hi(rk.y));
      const float4 k1 = make_float4(bf_lo(rk.z), bf_hi(rk.z), bf_lo(rk.w), bf_hi(rk.w));
      const float4 q0 = make_float4(bf_lo(rq.x), bf_hi(rq.x), bf_lo(rq.y), bf_hi(rq.y));
      const float4 q1 = make_float4(bf_lo(rq.z), bf_hi(rq.z), bf_lo(rq.w), bf_hi(rq.w));
      qk = fmaf(k0.x, q0.x, qk); qk = fmaf(k0.y, q0.y, qk);
      qk = fmaf(k0.z, q0.z, qk); qk = fmaf(k0.w, q0.w, qk);
      qk = fmaf(k1.x, q1.x, qk); qk = fmaf(k1.y, q1.y, qk);
      qk = fmaf(k1.z, q1.z, qk); qk = fmaf(k1.w, q1.w, qk);
      const int s0 = ((2 * p) ^ sw) * 16, s1 = ((2 * p + 1) ^ sw) * 16;
      *reinterpret_cast<float4*>(fs + kFK + tl * 512 + s0) = k0;
      *reinterpret_cast<float4*>(fs + kFK + tl * 512 + s1) = k1;
      *reinterpret_cast<float4*>(fs + kFQ + tl * 512 + s0) = q0;
      *reinterpret_cast<float4*>(fs + kFQ + tl * 512 + s1) = q1;
    }
    const uint4 rv = *reinterpret_cast<const uint4*>(rs + kRawV + tl * 64 + qd * 16);
    float4* dst = reinterpret_cast<float4*>(fs + kFV + tl * kCols * 4 + qd * 32);
    dst[0] = make_float4(bf_lo(rv.x), bf_hi(rv.x), bf_lo(rv.y), bf_hi(rv.y));
    dst[1] = make_float4(bf_lo(rv.z), bf_hi(rv.z), bf_lo(rv.w), bf_hi(rv.w));
  }
  qk += __shfl_xor_sync(0xffffffffu, qk, 1);
  qk += __shfl_xor_sync(0xffffffffu, qk, 2);
  if (live && qd == 0) {
    const float al = *reinterpret_cast<const float*>(rs + kRawA + tl * 4);
    const float be = *reinterpret_cast<const float*>(rs + kRawB + tl * 4);
    *reinterpret_cast<float4*>(fs + kFG + tl * 16) = make_float4(al, be, qk, 0.f);
  }
}

// Writes this warp's tokens of chunk cc (bf16 [kTc][32] outputs in os) to o: 16 bytes a lane.
__device__ __forceinline__ void stage_write_out(const ScanArgs& a, const uint8_t* os, int64_t cc,
                                                int h, int c0, int sw_warp, int lane) {
  const int tl = 8 * sw_warp + (lane >> 2), qd = lane & 3;
  if (tl >= chunk_tokens(a.T, cc)) return;
  uint8_t* dst = a.o + ((cc * kTc + tl) * a.H + h) * (int64_t)a.dv * 2 + (int64_t)c0 * 2;
  *reinterpret_cast<uint4*>(dst + qd * 16) = *reinterpret_cast<const uint4*>(os + tl * 64 + qd * 16);
}

// ---- consumer warps

__device__ __forceinline__ float2 f2(float x, float y) { return make_float2(x, y); }

struct TokenIn {
  float2 k[8], q[8];
  float v;
  float4 g;  // alpha, beta, k . q
};

// Token tt of the fp32 stage fs, as lane r of the group of column col needs it.
__device__ __forceinline__ void load_token(const uint8_t* fs, int tt, int r, int col, TokenIn& in) {
  const int sw = tt & 7;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int slot = ((r ^ sw) + 8 * c) * 16;
    const float4 kc = *reinterpret_cast<const float4*>(fs + kFK + tt * 512 + slot);
    const float4 qc = *reinterpret_cast<const float4*>(fs + kFQ + tt * 512 + slot);
    in.k[2 * c] = f2(kc.x, kc.y);
    in.k[2 * c + 1] = f2(kc.z, kc.w);
    in.q[2 * c] = f2(qc.x, qc.y);
    in.q[2 * c + 1] = f2(qc.z, qc.w);
  }
  in.v = *reinterpret_cast<const float*>(fs + kFV + (tt * kCols + col) * 4);
  in.g = *reinterpret_cast<const float4*>(fs + kFG + tt * 16);
}

// One token's step on a lane's 16 rows s (as 8 float pairs); returns o for the column.
__device__ __forceinline__ float token_step(float2 (&s)[8], const TokenIn& in) {
  float2 ra = __fmul2_rn(s[0], in.k[0]), rb = __fmul2_rn(s[1], in.k[1]);
  float2 pa = __fmul2_rn(s[0], in.q[0]), pb = __fmul2_rn(s[1], in.q[1]);
#pragma unroll
  for (int m = 1; m < 4; ++m) {
    ra = __ffma2_rn(s[2 * m], in.k[2 * m], ra);
    rb = __ffma2_rn(s[2 * m + 1], in.k[2 * m + 1], rb);
    pa = __ffma2_rn(s[2 * m], in.q[2 * m], pa);
    pb = __ffma2_rn(s[2 * m + 1], in.q[2 * m + 1], pb);
  }
  const float2 r2 = __fadd2_rn(ra, rb), p2 = __fadd2_rn(pa, pb);
  float r = r2.x + r2.y, p = p2.x + p2.y;
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) {  // the 8 lanes of the column's group
    r += __shfl_xor_sync(0xffffffffu, r, o);
    p += __shfl_xor_sync(0xffffffffu, p, o);
  }
  const float al = in.g.x, be = in.g.y, qk = in.g.z;
  const float u = be * (in.v - al * r);
  const float2 a2 = f2(al, al), u2 = f2(u, u);
#pragma unroll
  for (int m = 0; m < 8; ++m) s[m] = __ffma2_rn(in.k[m], u2, __fmul2_rn(s[m], a2));
  return fmaf(qk, u, al * p);
}

__global__ void __launch_bounds__(kThreads, 1) gdn_scan_kernel(ScanArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y, c0 = blockIdx.x * kCols;
  const int64_t nchunks = (a.T + kTc - 1) / kTc;
  uint8_t* raw = smem + kRawOff;
  uint8_t* fbuf = smem + kFOff;
  uint8_t* obuf = smem + kOOff;

  if (warp >= kCWarps) {  // staging warps
    const int sw_warp = warp - kCWarps;
    for (int c = 0; c < kRawStages; ++c)
      stage_issue(a, raw + c * kRawBytes, c, h, c0, sw_warp, lane);
    cp_async_wait2();
    __syncwarp();
    stage_convert(a, raw, fbuf, 0, sw_warp, lane);
    __syncthreads();
    for (int64_t cc = 0; cc < nchunks; ++cc) {
      // the raw stage of chunk cc was widened during the previous chunk: refill it
      stage_issue(a, raw + (cc % kRawStages) * kRawBytes, cc + kRawStages, h, c0, sw_warp, lane);
      cp_async_wait2();  // chunk cc + 1 has landed (this lane's copies)
      __syncwarp();      // ... and every lane's of this warp (each warp widens its own tokens)
      if (cc + 1 < nchunks)
        stage_convert(a, raw + ((cc + 1) % kRawStages) * kRawBytes,
                      fbuf + ((cc + 1) & 1) * kFBytes, cc + 1, sw_warp, lane);
      if (cc > 0) stage_write_out(a, obuf + ((cc - 1) & 1) * kOBytes, cc - 1, h, c0, sw_warp, lane);
      __syncthreads();
    }
    if (nchunks > 0)
      stage_write_out(a, obuf + ((nchunks - 1) & 1) * kOBytes, nchunks - 1, h, c0, sw_warp, lane);
    asm volatile("cp.async.wait_all;\n" ::: "memory");  // leave no copy in flight
    return;
  }

  // consumer: column col of the block, key rows 4 (r + 8 c) + e
  const int g = lane >> 3, r = lane & 7;
  const int col = 4 * warp + g;
  const int64_t sbase = (int64_t)h * kDk * a.dv + c0 + col;
  float2 s[8];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    float e[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      e[i] = a.s_in ? a.s_in[sbase + (int64_t)(4 * (r + 8 * c) + i) * a.dv] : 0.f;
    s[2 * c] = f2(e[0], e[1]);
    s[2 * c + 1] = f2(e[2], e[3]);
  }
  __syncthreads();  // chunk 0 staged
  for (int64_t cc = 0; cc < nchunks; ++cc) {
    const uint8_t* fs = fbuf + (cc & 1) * kFBytes;
    __nv_bfloat16* os = reinterpret_cast<__nv_bfloat16*>(obuf + (cc & 1) * kOBytes);
    const int n = (int)chunk_tokens(a.T, cc);
    // two token buffers in turn: the next token's inputs are read while this one computes
    // (slots past n hold stale values and are never used)
    TokenIn b0, b1;
    load_token(fs, 0, r, col, b0);
    int tt = 0;
    for (; tt + 1 < n; tt += 2) {
      load_token(fs, tt + 1, r, col, b1);
      const float o0 = token_step(s, b0);
      if (r == 0) os[tt * kCols + col] = __float2bfloat16_rn(o0);
      if (tt + 2 < kTc) load_token(fs, tt + 2, r, col, b0);
      const float o1 = token_step(s, b1);
      if (r == 0) os[(tt + 1) * kCols + col] = __float2bfloat16_rn(o1);
    }
    if (tt < n) {
      const float o0 = token_step(s, b0);
      if (r == 0) os[tt * kCols + col] = __float2bfloat16_rn(o0);
    }
    __syncthreads();
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const float e[4] = {s[2 * c].x, s[2 * c].y, s[2 * c + 1].x, s[2 * c + 1].y};
#pragma unroll
    for (int i = 0; i < 4; ++i) a.s_out[sbase + (int64_t)(4 * (r + 8 * c) + i) * a.dv] = e[i];
  }
}

bool misaligned(const void* p, uintptr_t m) { return (reinterpret_cast<uintptr_t>(p) & (m - 1)) != 0; }

}  // namespace

extern "C" int gdn_scan(const void* q, const void* k, const void* v, const float* alpha,
                        const float* beta, const float* state_in, float* state_out, void* o,
                        int64_t T, int H, int dk, int dv, void* stream) {
  if (T < 0 || H < 1 || !state_out) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!q || !k || !v || !alpha || !beta || !o)) return MOE_ERR_INVALID_ARG;
  if (dk != kDk || dv < kCols || dv % kCols || dv > 4096 || H > 65535) return MOE_ERR_UNSUPPORTED;
  if (misaligned(state_out, 4) || (state_in && misaligned(state_in, 4))) return MOE_ERR_ALIGNMENT;
  if (T > 0 && (misaligned(q, 16) || misaligned(k, 16) || misaligned(v, 16) || misaligned(o, 16) ||
                misaligned(alpha, 4) || misaligned(beta, 4)))
    return MOE_ERR_ALIGNMENT;
  if (cudaFuncSetAttribute(gdn_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmemBytes) != cudaSuccess ||
      cudaFuncSetAttribute(gdn_scan_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared) != cudaSuccess)
    return MOE_ERR_CUDA;
  ScanArgs a{static_cast<const uint8_t*>(q), static_cast<const uint8_t*>(k),
             static_cast<const uint8_t*>(v), alpha, beta, state_in, state_out,
             static_cast<uint8_t*>(o), T, H, dv};
  gdn_scan_kernel<<<dim3(dv / kCols, H), kThreads, kSmemBytes, static_cast<cudaStream_t>(stream)>>>(a);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
