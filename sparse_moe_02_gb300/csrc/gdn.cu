// Gated DeltaNet recurrent scan (include/gdn.h states the rule, layouts and errors).
//
// "Optimizing on-device inference for Apple Silicon", § "Keep recurrent state on chip": a group
// of lanes per state column, the column held in registers for the whole scan, partial sums
// exchanged between lanes by shuffles, the state written back once at the end.
//
// GB300 layout of the work: a block owns one head and 32 value columns (grid: dv/32 x H).
// Eight consumer warps (two per scheduler, so that one warp's waits on shuffles and dependent
// arithmetic are covered by the other's work) hold the 32 columns, four per warp: the 16 lanes of
// a group own two adjacent columns, lane r holding the 8 key rows 4(r + 16c) + e (c < 2, e < 4)
// of both as fp32 registers.  Two columns per lane halve the shared-memory reads of k and q per
// state element (every lane reads its rows of k and q per token, whatever its column count).
//
// Per token t the lane needs r_t = S_{t-1}^T k_t and p_t = S_{t-1}^T q_t, complete sums over the
// 128 rows: four halving exchange rounds over the group leave each lane one of the four sums
// (k or q, column 0 or 1); the k-lanes form u_t and two shuffles hand it to the whole group.  To keep those rounds off the token-to-token
// chain, the dot products are taken one token early, against the state before the previous
// token's update, and corrected by a scalar (S_{t-1} = alpha_{t-1} S_{t-2} + k_{t-1} u_{t-1}^T):
//   r_t = alpha_{t-1} (S_{t-2}^T k_t) + (k_{t-1} . k_t) u_{t-1}
//   p_t = alpha_{t-1} (S_{t-2}^T q_t) + (k_{t-1} . q_t) u_{t-1}
// so while token t's update runs, the sums for token t + 1 are in flight.  The first token of
// every 32-token chunk takes its sums directly (no correction).  Then
//   u_t = beta_t (v_t - alpha_t r_t),  o_t = alpha_t p_t + (k_t . q_t) u_t,
//   S_t = alpha_t S_{t-1} + k_t u_t^T.
//
// Four staging warps (one per scheduler) feed the consumers: chunks of 32 tokens' k, q (one
// head), v (the block's 32 columns) and gates come in by cp.async two chunks ahead; the consumers
// read k and q there as bf16 (half the shared-memory traffic of fp32, widened on the integer
// pipe), while the staging warps form the per-token dot products k_t . q_t, k_{t-1} . k_t and
// k_{t-1} . q_t and widen v and the gates into one of two fp32 chunk buffers; the outputs the
// consumers leave in shared memory go out in 64-byte rows.  One block barrier per chunk hands
// the buffers over; nothing waits on a flag, so nothing can hang.
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
constexpr int kRawStages = 3;                 // bf16 chunks: read, landed, in flight

// Shared memory, bytes.
//   raw stage: k, q [kTc][256] (16-byte piece p of token t at slot p ^ (t & 7)); kprev [4][256]
//     (staging warp w's copy of the k row of token 8w - 1, plain order); v [kTc][64]; alpha,
//     beta [kTc];
//   fp32 stage: v [kTc][32]; gates [kTc][8] = (alpha, beta, k.q, k_prev.k, k_prev.q, 0, 0, 0);
//   output stage: [kTc][32] bf16.
// The xor swizzle keeps the staging warps' per-token rows and the consumers' reads (16 lanes,
// 128 consecutive bytes of k or q) free of bank conflicts.
constexpr int kRawK = 0;
constexpr int kRawQ = kRawK + kTc * 256;
constexpr int kRawKp = kRawQ + kTc * 256;
constexpr int kRawV = kRawKp + kSWarps * 256;
constexpr int kRawA = kRawV + kTc * 64;
constexpr int kRawB = kRawA + kTc * 4;
constexpr int kRawBytes = kRawB + kTc * 4;
constexpr int kFV = 0;
constexpr int kFG = kFV + kTc * kCols * 4;
constexpr int kFBytes = kFG + kTc * 32;
constexpr int kOBytes = kTc * kCols * 2;
constexpr int kRawOff = 0;
constexpr int kFOff = kRawOff + kRawStages * kRawBytes;
constexpr int kOOff = kFOff + 2 * kFBytes;
constexpr int kSmemBytes = kOOff + 2 * kOBytes;
static_assert(kRawBytes % 16 == 0 && kFBytes % 16 == 0 && kOBytes % 16 == 0, "16-byte stages");
static_assert(kTc == 8 * kSWarps, "each staging warp owns 8 tokens of a chunk");

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

// At most one group of this thread still pending.
__device__ __forceinline__ void cp_async_wait1() {
  asm volatile("cp.async.wait_group 1;\n" ::: "memory");
}

// bf16 pairs of a 32-bit word -> fp32 (exact): element 2m in the low half.
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void widen8(uint4 w, float (&f)[8]) {
  f[0] = bf_lo(w.x); f[1] = bf_hi(w.x); f[2] = bf_lo(w.y); f[3] = bf_hi(w.y);
  f[4] = bf_lo(w.z); f[5] = bf_hi(w.z); f[6] = bf_lo(w.w); f[7] = bf_hi(w.w);
}

__device__ __forceinline__ int64_t chunk_tokens(int64_t T, int64_t cc) {
  const int64_t left = T - cc * kTc;
  return left <= 0 ? 0 : (left < kTc ? left : kTc);
}

// ---- staging warps
//
// Staging warp w (one per SM sub-partition, so that the staging work is spread evenly over the
// four schedulers) owns tokens 8w .. 8w + 7 of every chunk: it copies their inputs (and the k row
// of token 8w - 1, for k_{t-1} . k_t), widens them and writes their outputs.  In the widening
// and the write-out, lane l works on token 8w + l / 4, quarter l % 4 of the row.

// cp.async of this warp's tokens of chunk cc into raw stage rs (one commit group, empty past
// the end of the prompt).
__device__ __forceinline__ void stage_issue(const ScanArgs& a, uint8_t* rs, int64_t cc, int h,
                                            int c0, int w, int lane) {
  const int64_t n = chunk_tokens(a.T, cc);
  const int64_t t0 = cc * kTc;
#pragma unroll
  for (int it = 0; it < 4; ++it) {  // two tokens' 256-byte k and q rows per instruction
    const int tl = 8 * w + 2 * it + (lane >> 4), p = lane & 15;
    if (tl < n) {
      const int64_t row = ((t0 + tl) * a.H + h) * (kDk * 2);
      const int slot = (p ^ (tl & 7)) * 16;
      cp_async16(rs + kRawK + tl * 256 + slot, a.k + row + p * 16);
      cp_async16(rs + kRawQ + tl * 256 + slot, a.q + row + p * 16);
    }
  }
  if (w > 0 && lane < 16 && 8 * w < n) {  // k of token 8w - 1 (owned by the warp before)
    const int64_t row = ((t0 + 8 * w - 1) * a.H + h) * (kDk * 2);
    cp_async16(rs + kRawKp + w * 256 + lane * 16, a.k + row + lane * 16);
  }
  {  // eight tokens' 64-byte v slices
    const int tl = 8 * w + (lane >> 2), pc = lane & 3;
    if (tl < n)
      cp_async16(rs + kRawV + tl * 64 + pc * 16,
                 a.v + ((t0 + tl) * a.H + h) * (int64_t)a.dv * 2 + (int64_t)c0 * 2 + pc * 16);
  }
  if (lane < 8 && 8 * w + lane < n) {
    const int tl = 8 * w + lane;
    cp_async4(rs + kRawA + tl * 4, a.alpha + (t0 + tl) * a.H + h);
    cp_async4(rs + kRawB + tl * 4, a.beta + (t0 + tl) * a.H + h);
  }
  cp_async_commit();
}

// Widens this warp's tokens' v and gates of chunk cc from raw stage rs into fp32 stage fs, with
// the dot products k_t . q_t, k_{t-1} . k_t and k_{t-1} . q_t of each token (zero for the chunk's first
// token, which does not use them): each lane sums its quarter of the rows (32 products in
// ascending index), then the four quarters are added by two xor shuffles, the same tree in every
// lane.
__device__ __forceinline__ void stage_convert(const ScanArgs& a, const uint8_t* rs, uint8_t* fs,
                                              int64_t cc, int w, int lane) {
  const int tl = 8 * w + (lane >> 2), qd = lane & 3;
  const bool live = tl < chunk_tokens(a.T, cc);
  const int sw = tl & 7;
  float qk = 0.f, kk = 0.f, kq = 0.f;
  if (live) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int p = 4 * qd + i;
      float k8[8], q8[8], kp8[8];
      widen8(*reinterpret_cast<const uint4*>(rs + kRawK + tl * 256 + (p ^ sw) * 16), k8);
      widen8(*reinterpret_cast<const uint4*>(rs + kRawQ + tl * 256 + (p ^ sw) * 16), q8);
      if (tl == 0)
#pragma unroll
        for (int e = 0; e < 8; ++e) kp8[e] = 0.f;
      else if (tl == 8 * w)
        widen8(*reinterpret_cast<const uint4*>(rs + kRawKp + w * 256 + p * 16), kp8);
      else
        widen8(*reinterpret_cast<const uint4*>(rs + kRawK + (tl - 1) * 256 +
                                               (p ^ ((tl - 1) & 7)) * 16), kp8);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        qk = fmaf(k8[e], q8[e], qk);
        kk = fmaf(kp8[e], k8[e], kk);
        kq = fmaf(kp8[e], q8[e], kq);
      }
    }
    float v8[8];
    widen8(*reinterpret_cast<const uint4*>(rs + kRawV + tl * 64 + qd * 16), v8);
    float4* dst = reinterpret_cast<float4*>(fs + kFV + tl * kCols * 4 + qd * 32);
    dst[0] = make_float4(v8[0], v8[1], v8[2], v8[3]);
    dst[1] = make_float4(v8[4], v8[5], v8[6], v8[7]);
  }
#pragma unroll
  for (int o = 1; o < 4; o <<= 1) {
    qk += __shfl_xor_sync(0xffffffffu, qk, o);
    kk += __shfl_xor_sync(0xffffffffu, kk, o);
    kq += __shfl_xor_sync(0xffffffffu, kq, o);
  }
  if (live && qd == 0) {
    const float al = *reinterpret_cast<const float*>(rs + kRawA + tl * 4);
    const float be = *reinterpret_cast<const float*>(rs + kRawB + tl * 4);
    float4* g = reinterpret_cast<float4*>(fs + kFG + tl * 32);
    g[0] = make_float4(al, be, qk, kk);
    g[1] = make_float4(kq, 0.f, 0.f, 0.f);
  }
}

// Writes this warp's tokens of chunk cc (bf16 [kTc][32] outputs in os) to o: 16 bytes a lane.
__device__ __forceinline__ void stage_write_out(const ScanArgs& a, const uint8_t* os, int64_t cc,
                                                int h, int c0, int w, int lane) {
  const int tl = 8 * w + (lane >> 2), qd = lane & 3;
  if (tl >= chunk_tokens(a.T, cc)) return;
  uint8_t* dst = a.o + ((cc * kTc + tl) * a.H + h) * (int64_t)a.dv * 2 + (int64_t)c0 * 2;
  *reinterpret_cast<uint4*>(dst + qd * 16) = *reinterpret_cast<const uint4*>(os + tl * 64 + qd * 16);
}

// ---- consumer warps

__device__ __forceinline__ float2 f2(float x, float y) { return make_float2(x, y); }

struct KQ {
  float2 k[4], q[4];
};

// A token's k and q at the lane's 8 rows 4(r + 16c) + e, as row pairs (e = 0, 1 and e = 2, 3),
// read as bf16 from raw stage rs: the rows 64c + 4r .. 64c + 4r + 3 are 8 bytes at offset
// 8 (r & 1) of the 16-byte piece (r >> 1) + 8c of the token's row.
__device__ __forceinline__ void load_kq(const uint8_t* rs, int tt, int r, KQ& x) {
  const int sw = tt & 7;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int off = tt * 256 + ((((r >> 1) + 8 * c) ^ sw) * 16) + (r & 1) * 8;
    const uint2 kw = *reinterpret_cast<const uint2*>(rs + kRawK + off);
    const uint2 qw = *reinterpret_cast<const uint2*>(rs + kRawQ + off);
    x.k[2 * c] = f2(bf_lo(kw.x), bf_hi(kw.x));
    x.k[2 * c + 1] = f2(bf_lo(kw.y), bf_hi(kw.y));
    x.q[2 * c] = f2(bf_lo(qw.x), bf_hi(qw.x));
    x.q[2 * c + 1] = f2(bf_lo(qw.y), bf_hi(qw.y));
  }
}

// d = (S^T k, S^T q) of both columns over the lane's rows: d[j] = k-sum of column j,
// d[2 + j] = q-sum.
__device__ __forceinline__ void group_dots(const float2 (&s)[2][4], const KQ& x, float (&d)[4]) {
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    float2 ka = __fmul2_rn(s[j][0], x.k[0]), kb = __fmul2_rn(s[j][1], x.k[1]);
    float2 qa = __fmul2_rn(s[j][0], x.q[0]), qb = __fmul2_rn(s[j][1], x.q[1]);
    ka = __ffma2_rn(s[j][2], x.k[2], ka);
    kb = __ffma2_rn(s[j][3], x.k[3], kb);
    qa = __ffma2_rn(s[j][2], x.q[2], qa);
    qb = __ffma2_rn(s[j][3], x.q[3], qb);
    const float2 k2 = __fadd2_rn(ka, kb), q2 = __fadd2_rn(qa, qb);
    d[j] = k2.x + k2.y;
    d[2 + j] = q2.x + q2.y;
  }
}

// Sums d over the group's 16 lanes by halving exchanges: after the four rounds lane r holds one
// full sum, the k-sum (r < 8) or q-sum (r >= 8) of column (r >> 2) & 1 (the four lanes that
// differ only in bits 0 and 1 hold the same).  Five shuffles instead of sixteen; the additions
// form the same tree in every lane that holds a given sum, so the result does not depend on
// which lane holds it.
__device__ __forceinline__ float group_sum_split(const float (&d)[4], int r) {
  const bool hi = (r & 8) != 0;  // keeps the q-sums
  const float s0 = hi ? d[0] : d[2], s1 = hi ? d[1] : d[3];
  float k0 = hi ? d[2] : d[0], k1 = hi ? d[3] : d[1];
  k0 += __shfl_xor_sync(0xffffffffu, s0, 8);
  k1 += __shfl_xor_sync(0xffffffffu, s1, 8);
  const bool c1 = (r & 4) != 0;  // keeps column 1
  const float snd = c1 ? k0 : k1;
  float x = c1 ? k1 : k0;
  x += __shfl_xor_sync(0xffffffffu, snd, 4);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  return x;
}

// Carried from one token to the next, per lane: the full sum this lane holds (S_{t-2}^T k_t or
// S_{t-2}^T q_t of its column; for the chunk's first token, S_{t-1}^T k_t or q_t with
// al_prev = 1 and u_prev = 0), alpha_{t-1} and u_{t-1} of both columns.
struct Carry {
  float x;
  float al_prev;
  float u_prev[2];
};

// Token tt of the chunk in fs: cur holds its k (for the update), nxt the next token's k and q
// (for the early sums, when has_next).  Lanes r = 8 + 4j end with o_t of column j in *o.
__device__ __forceinline__ void token_step(float2 (&s)[2][4], Carry& cy, const uint8_t* fs,
                                           int tt, int col0, int r, const KQ& cur, const KQ& nxt,
                                           bool has_next, float* o) {
  const float4 g0 = *reinterpret_cast<const float4*>(fs + kFG + tt * 32);
  const float kq = *reinterpret_cast<const float*>(fs + kFG + tt * 32 + 16);
  const int j = (r >> 2) & 1;
  const bool isq = r >= 8;
  const float vj = *reinterpret_cast<const float*>(fs + kFV + (tt * kCols + col0 + j) * 4);
  const float al = g0.x, be = g0.y, qk = g0.z, kk = g0.w;
  float d[4];
  if (has_next) group_dots(s, nxt, d);  // against S_{t-1}, before this token's update
  // this lane's sum: r_t (k-lanes) or p_t (q-lanes) of column j
  const float up = j ? cy.u_prev[1] : cy.u_prev[0];
  const float x = fmaf(isq ? kq : kk, up, cy.al_prev * cy.x);
  const float uc = be * (vj - al * x);  // u_t of column j on the k-lanes
  const float u0 = __shfl_sync(0xffffffffu, uc, (threadIdx.x & 16) | 0);
  const float u1 = __shfl_sync(0xffffffffu, uc, (threadIdx.x & 16) | 4);
  *o = fmaf(qk, j ? u1 : u0, al * x);  // o_t of column j on the q-lanes
  const float2 a2 = f2(al, al), w0 = f2(u0, u0), w1 = f2(u1, u1);
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    s[0][m] = __ffma2_rn(cur.k[m], w0, __fmul2_rn(s[0][m], a2));
    s[1][m] = __ffma2_rn(cur.k[m], w1, __fmul2_rn(s[1][m], a2));
  }
  if (has_next) cy.x = group_sum_split(d, r);
  cy.al_prev = al;
  cy.u_prev[0] = u0;
  cy.u_prev[1] = u1;
}

// Lanes 8 and 12 of the group hold o_t of columns 0 and 1.
__device__ __forceinline__ void store_o(uint8_t* os, int tt, int col0, int r, float o) {
  if (r == 8 || r == 12)
    *reinterpret_cast<__nv_bfloat16*>(os + (tt * kCols + col0 + ((r >> 2) & 1)) * 2) =
        __float2bfloat16_rn(o);
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
    const int w = warp - kCWarps;
    for (int c = 0; c < 2; ++c) stage_issue(a, raw + c * kRawBytes, c, h, c0, w, lane);
    cp_async_wait1();
    __syncwarp();
    stage_convert(a, raw, fbuf, 0, w, lane);
    __syncthreads();
    for (int64_t cc = 0; cc < nchunks; ++cc) {
      // the consumers read chunk cc's raw stage; the stage of chunk cc - 1 is free again
      stage_issue(a, raw + ((cc + 2) % kRawStages) * kRawBytes, cc + 2, h, c0, w, lane);
      cp_async_wait1();  // chunk cc + 1 has landed (this lane's copies; the block barrier below
      __syncwarp();      // makes every lane's visible to the consumers)
      if (cc + 1 < nchunks)
        stage_convert(a, raw + ((cc + 1) % kRawStages) * kRawBytes,
                      fbuf + ((cc + 1) & 1) * kFBytes, cc + 1, w, lane);
      if (cc > 0) stage_write_out(a, obuf + ((cc - 1) & 1) * kOBytes, cc - 1, h, c0, w, lane);
      __syncthreads();
    }
    if (nchunks > 0)
      stage_write_out(a, obuf + ((nchunks - 1) & 1) * kOBytes, nchunks - 1, h, c0, w, lane);
    asm volatile("cp.async.wait_all;\n" ::: "memory");  // leave no copy in flight
    return;
  }

  // consumer: columns col0, col0 + 1 of the block, key rows 4 (r + 16 c) + e
  const int g = lane >> 4, r = lane & 15;
  const int col0 = 4 * warp + 2 * g;
  const int64_t sbase = (int64_t)h * kDk * a.dv + c0 + col0;
  float2 s[2][4];
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      float2 e0 = f2(0.f, 0.f), e1 = f2(0.f, 0.f);  // rows 4P + 2i and 4P + 2i + 1, both columns
      if (a.s_in) {
        const int row = 4 * (r + 16 * c) + 2 * i;
        e0 = *reinterpret_cast<const float2*>(a.s_in + sbase + (int64_t)row * a.dv);
        e1 = *reinterpret_cast<const float2*>(a.s_in + sbase + (int64_t)(row + 1) * a.dv);
      }
      s[0][2 * c + i] = f2(e0.x, e1.x);
      s[1][2 * c + i] = f2(e0.y, e1.y);
    }
  __syncthreads();  // chunk 0 staged
  for (int64_t cc = 0; cc < nchunks; ++cc) {
    const uint8_t* fs = fbuf + (cc & 1) * kFBytes;
    const uint8_t* rs = raw + (cc % kRawStages) * kRawBytes;
    uint8_t* os = obuf + (cc & 1) * kOBytes;
    const int n = (int)chunk_tokens(a.T, cc);
    // the chunk's first token: its sums taken directly from the current state
    KQ x0, x1;
    load_kq(rs, 0, r, x0);
    Carry cy;
    {
      float d[4];
      group_dots(s, x0, d);
      cy.x = group_sum_split(d, r);
      cy.al_prev = 1.f;
      cy.u_prev[0] = cy.u_prev[1] = 0.f;
    }
    load_kq(rs, 1, r, x1);  // slot 1 exists even when n == 1 (stale, unused)
    // two buffers in turn: x0 holds the even token's k and q, x1 the odd one's
    int tt = 0;
    float o;
    for (; tt + 1 < n; tt += 2) {
      token_step(s, cy, fs, tt, col0, r, x0, x1, true, &o);
      store_o(os, tt, col0, r, o);
      if (tt + 2 < kTc) load_kq(rs, tt + 2, r, x0);
      token_step(s, cy, fs, tt + 1, col0, r, x1, x0, tt + 2 < n, &o);
      store_o(os, tt + 1, col0, r, o);
      if (tt + 3 < kTc) load_kq(rs, tt + 3, r, x1);
    }
    if (tt < n) {
      token_step(s, cy, fs, tt, col0, r, x0, x1, false, &o);
      store_o(os, tt, col0, r, o);
    }
    __syncthreads();
  }
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int row = 4 * (r + 16 * c) + 2 * i;
      *reinterpret_cast<float2*>(a.s_out + sbase + (int64_t)row * a.dv) =
          f2(s[0][2 * c + i].x, s[1][2 * c + i].x);
      *reinterpret_cast<float2*>(a.s_out + sbase + (int64_t)(row + 1) * a.dv) =
          f2(s[0][2 * c + i].y, s[1][2 * c + i].y);
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
  if (misaligned(state_out, 8) || (state_in && misaligned(state_in, 8))) return MOE_ERR_ALIGNMENT;
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
  // the launch's own status (not cudaGetLastError, which would also take and clear an earlier,
  // unrelated error)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(dv / kCols, H);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = static_cast<cudaStream_t>(stream);
  return cudaLaunchKernelEx(&cfg, gdn_scan_kernel, a) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
