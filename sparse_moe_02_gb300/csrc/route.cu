// Routing chain of the MoE layer on the GPU ("Optimizing on-device inference for Apple
// Silicon", § "Keep expert routing on the GPU"): router scores and top-8 selection, a
// histogram of assignments per expert, a prefix scan into start offsets, a scatter of the
// rows into their expert groups, and the block map (work units) of the grouped GEMMs.
// Nothing here waits for the host, and every result is deterministic: the histogram is
// kept per 128-token block and combined in block order, and ranks inside a block come
// from bit masks in token order, so no atomic ordering reaches an output.
#include "layer.cuh"
#include "plan.cuh"
#include "ptx.cuh"
#include "select.cuh"

namespace moe {
namespace {

// ---------------------------------------------------------------- router GEMM + top-8

// A cluster of four blocks per 128 tokens splits the reduction: block r multiplies the
// k-blocks r, r + 4, r + 8, ... of x and the router matrix (tcgen05, M = 128 tokens, N = 256
// experts) into a partial logit tile in TMEM, so each block streams a quarter of the tile's
// inputs.  The partials are summed in the block that owns the tokens: TMEM lane quadrant q
// (tokens 32q .. 32q + 31) belongs to block q.  Each block writes its three foreign quadrants
// to shared memory and sends each to its owner with one bulk copy (distributed shared memory,
// completing on the owner's mbarrier); the owner adds the four partials in block order and
// selects each token's top 8 with eight threads per token.
constexpr int kRtCluster = 4;
constexpr int kRtStages = 4;
constexpr int kRtA = kBlockTokens * kBK * 2;          // x tile: 128 tokens x 64 (16 KB)
constexpr int kRtB = kE * kBK * 2;                    // router tile: 256 experts x 64 (32 KB)
constexpr int kRtStage = kRtA + kRtB;
constexpr int kRtThreads = 320;                       // producer, MMA, 8 epilogue warps
constexpr int kRtTok = kBlockTokens / kRtCluster;     // tokens owned per block
constexpr int kRtSlot = kRtTok * kE * 4;              // one quadrant of partial logits (32 KB)
// after the ring drains: received partials [4 source blocks] then outgoing quadrants [3]
constexpr int kRtRecv = 0, kRtSend = kRtCluster * kRtSlot;
constexpr int kRtArea = kRtSend + (kRtCluster - 1) * kRtSlot;
constexpr int kRtBody = kRtArea > kRtStages * kRtStage ? kRtArea : kRtStages * kRtStage;
constexpr int kRtSmem = kRtBody + 1024 + 2048;

// Float e of token row `row` in a quadrant slot: rows of 256 floats whose 16-byte chunks are
// XOR-swizzled by the row, so that a warp writing one chunk of 32 rows, or reading chunks of a
// few rows, spreads over all banks.
__device__ __forceinline__ float* slot_at(float* slot, int row, int e) {
  return slot + row * kE + ((((e >> 2) ^ (row & 7))) << 2) + (e & 3);
}

struct RouterArgs {
  const float* bias;
  int T, d;
  int32_t* topk_idx;
  float* topk_w;
  int32_t* hist;
  int* err;
};

// Inserts (x, e) into the descending list v/id (8 entries) when it ranks above the last one.
// Values arrive with ascending e, so an equal value stays behind the entries already held.
// The eight comparisons are independent (collected as bits: held as an array of bools, this
// was miscompiled by nvcc 13.0 once fully unrolled); each slot then takes its own value, its
// upper neighbour's or x.
__device__ __forceinline__ void top8_insert(float (&v)[8], int (&id)[8], float x, int e) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) m |= (x > v[i] ? 1u : 0u) << i;
#pragma unroll
  for (int i = 7; i > 0; --i) {
    const bool ci = (m >> i) & 1u, cp = (m >> (i - 1)) & 1u;
    v[i] = ci ? (cp ? v[i - 1] : x) : v[i];
    id[i] = ci ? (cp ? id[i - 1] : e) : id[i];
  }
  if (m & 1u) {
    v[0] = x;
    id[0] = e;
  }
}

__global__ void __launch_bounds__(kRtThreads, 1)
    router_topk_kernel(const __grid_constant__ CUtensorMap tm_x,
                       const __grid_constant__ CUtensorMap tm_wr, RouterArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  float* recv = reinterpret_cast<float*>(smem + kRtRecv);  // [src block] slots, after the ring
  float* send = reinterpret_cast<float*>(smem + kRtSend);  // [3] outgoing quadrants
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kRtBody);
  uint64_t* empty = full + kRtStages;
  uint64_t* tfull = empty + kRtStages;
  uint64_t* rfull = tfull + 1;  // the three foreign partials of this block's tokens arrived
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(rfull + 1);
  int* hist_s = reinterpret_cast<int*>(tmem_slot + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int blk = (int)cluster_id_x();  // 128-token block
  const int KB = a.d / kBK;
  const int nk = KB > (int)rank ? (KB - (int)rank + kRtCluster - 1) / kRtCluster : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRtStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(rfull, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(rfull, (kRtCluster - 1) * kRtSlot);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kE);
    tmem_relinquish();
  }
  for (int i = threadIdx.x; i < kE; i += blockDim.x) hist_s[i] = 0;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // x (and the bias) may come from the previous kernel on the stream

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tensormap(&tm_x);
      prefetch_tensormap(&tm_wr);
      const uint64_t keep = policy_evict_last();  // x is gathered again by the expert GEMMs
      int stage = 0;
      uint32_t ph = 0;
      for (int i = 0; i < nk; ++i) {
        const int kb = (int)rank + kRtCluster * i;
        if (!mbar_wait(&empty[stage], ph ^ 1, a.err)) break;
        uint8_t* st = smem + stage * kRtStage;
        mbar_arrive_expect_tx(&full[stage], kRtStage);
        tma_load_2d(st, &tm_x, &full[stage], kb * kBK, blk * kBlockTokens, keep);
        tma_load_2d(st + kRtA, &tm_wr, &full[stage], kb * kBK, 0, keep);
        if (++stage == kRtStages) { stage = 0; ph ^= 1; }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && nk > 0) {
      const uint32_t idesc = idesc_bf16(128, kE);
      int stage = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int i = 0; i < nk; ++i) {
        if (!mbar_wait(&full[stage], ph, a.err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + stage * kRtStage), sb = sa + kRtA;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          mma_bf16(tmem, sdesc_k128(sa + kk * 32), sdesc_k128(sb + kk * 32), idesc,
                   (i | kk) != 0);
        mma_commit(&empty[stage]);
        if (++stage == kRtStages) { stage = 0; ph ^= 1; }
      }
      if (ok) mma_commit(tfull);
    }
  }
  // epilogue: TMEM quadrant q to the local slot of block q's partial (its own quadrant straight
  // into the receive slot); after the cluster barrier every block's ring has drained, so the
  // foreign quadrants may be copied into their owners' receive slots
  if (warp >= 2) {
    const int q = warp & 3, half = (warp - 2) >> 2;
    const bool have = nk == 0 || mbar_wait(tfull, 0, a.err);
    tc_fence_after();
    float* dst = q == (int)rank ? recv + (int)rank * (kRtSlot / 4)
                                : send + ((q - (int)rank + kRtCluster - 1) & 3) * (kRtSlot / 4);
    uint32_t r[128];
    if (nk > 0 && have) {
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 16)
        tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(half * 128 + c0),
                  *reinterpret_cast<uint32_t(*)[16]>(r + c0));
      tmem_wait_ld();
    } else {
#pragma unroll
      for (int i = 0; i < 128; ++i) r[i] = 0u;
    }
#pragma unroll
    for (int j = 0; j < 32; ++j)
      *reinterpret_cast<uint4*>(slot_at(dst, lane, half * 128 + 4 * j)) =
          make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
    fence_proxy_async_smem();  // read next by the bulk copies
  }
  tc_fence_before();
  cluster_sync();
  if (warp >= 2 && warp < 2 + kRtCluster - 1 && lane == 0) {
    const int s = warp - 2, q = ((int)rank + 1 + s) & 3;
    bulk_s2cluster(map_shared(recv + (int)rank * (kRtSlot / 4), q), send + s * (kRtSlot / 4),
                   kRtSlot, map_shared(rfull, q));
    bulk_commit();
  }

  if (warp >= 2) {
    // select: thread (token tl, part p) takes experts 4p + 32i + j (i < 8, j < 4).  The sums
    // go back into receive slot 0 (each thread owns those words).  Any value below
    // tau = min over the 8 parts of the part's largest value has at least 8 values of the token
    // above it, so only values >= tau are inserted: a few per thread, taken one at a time.
    const int tid = threadIdx.x - 64, tl = tid >> 3, p = tid & 7;
    const int t = blk * kBlockTokens + (int)rank * kRtTok + tl;
    mbar_wait(rfull, 0, a.err);
    float sv[32];
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e0 = 4 * p + 32 * i;
      float4 s = *reinterpret_cast<const float4*>(slot_at(recv, tl, e0));
#pragma unroll
      for (int src = 1; src < kRtCluster; ++src) {
        const float4 u =
            *reinterpret_cast<const float4*>(slot_at(recv + src * (kRtSlot / 4), tl, e0));
        s.x += u.x; s.y += u.y; s.z += u.z; s.w += u.w;
      }
      if (a.bias) {
        const float4 bb = __ldg(reinterpret_cast<const float4*>(a.bias + e0));
        s.x += bb.x; s.y += bb.y; s.z += bb.z; s.w += bb.w;
      }
      *reinterpret_cast<float4*>(slot_at(recv, tl, e0)) = s;
      sv[4 * i] = s.x; sv[4 * i + 1] = s.y; sv[4 * i + 2] = s.z; sv[4 * i + 3] = s.w;
      mx = fmaxf(mx, fmaxf(fmaxf(s.x, s.y), fmaxf(s.z, s.w)));
    }
    float tau = mx;
    tau = fminf(tau, __shfl_xor_sync(0xffffffffu, tau, 1));
    tau = fminf(tau, __shfl_xor_sync(0xffffffffu, tau, 2));
    tau = fminf(tau, __shfl_xor_sync(0xffffffffu, tau, 4));
    uint32_t pass = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) pass |= (sv[j] >= tau ? 1u : 0u) << j;
    float v[8];
    int id[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) { v[i] = -INFINITY; id[i] = 0x7fffffff; }
    while (__any_sync(0xffffffffu, pass != 0)) {
      if (pass) {
        const int j = __ffs(pass) - 1;  // ascending j: ascending expert id
        pass &= pass - 1;
        const int e = 4 * p + 32 * (j >> 2) + (j & 3);
        top8_insert(v, id, *slot_at(recv, tl, e), e);
      }
    }
    top8_merge_xor(v, id, 1);
    top8_merge_xor(v, id, 2);
    top8_merge_xor(v, id, 4);
    if (p == 0 && t < a.T) {
      // list the kept experts in ascending id; softmax over the kept logits
#pragma unroll
      for (int i = 0; i < 7; ++i)
#pragma unroll
        for (int j = 0; j < 7 - i; ++j)
          if (id[j] > id[j + 1]) {
            int ti = id[j]; id[j] = id[j + 1]; id[j + 1] = ti;
            float tv = v[j]; v[j] = v[j + 1]; v[j + 1] = tv;
          }
      float mx = v[0];
#pragma unroll
      for (int j = 1; j < 8; ++j) mx = fmaxf(mx, v[j]);
      float ex[8], sum = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) { ex[j] = __expf(v[j] - mx); sum += ex[j]; }
      int4* pi = reinterpret_cast<int4*>(a.topk_idx + (size_t)t * kTopK);
      float4* pw = reinterpret_cast<float4*>(a.topk_w + (size_t)t * kTopK);
      pi[0] = make_int4(id[0], id[1], id[2], id[3]);
      pi[1] = make_int4(id[4], id[5], id[6], id[7]);
      pw[0] = make_float4(ex[0] / sum, ex[1] / sum, ex[2] / sum, ex[3] / sum);
      pw[1] = make_float4(ex[4] / sum, ex[5] / sum, ex[6] / sum, ex[7] / sum);
#pragma unroll
      for (int j = 0; j < 8; ++j) red_cluster_add(map_shared(hist_s + id[j], 0), 1);
    }
  }
  if (warp >= 2 && warp < 2 + kRtCluster - 1 && lane == 0) bulk_wait_read();  // sources free
  cluster_sync();  // the leader's histogram is complete
  if (rank == 0 && warp >= 2) {
    const int e = threadIdx.x - 64;
    a.hist[(size_t)blk * kE + e] = hist_s[e];
  }
  pdl_trigger();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kE);
}

// Plan and scatter in one launch, one block of 256 threads per 128-token block (used while
// the token blocks are few, so that every block can afford to read the whole histogram):
// thread e sums expert e's counts over all token blocks (the total) and over the blocks before
// this one (its scatter base); every block builds the same group table, writes its share of
// the unit lists and scatters its own tokens; block 0 writes the global plan outputs.
__global__ void __launch_bounds__(256)
    route_plan_scatter_kernel(PlanArgs p, const int32_t* topk_idx, int32_t* perm, RouteWs ws) {
  __shared__ GroupTable G;
  __shared__ int s_pre[kE];
  __shared__ uint32_t mask[4][kE];
  pdl_wait();
  const int e = threadIdx.x, blk = blockIdx.x;
  int pre = 0, tot = 0;
  for (int b0 = 0; b0 < p.nblk; b0 += 32) {
    int c[32];
#pragma unroll
    for (int i = 0; i < 32; ++i)
      c[i] = b0 + i < p.nblk ? __ldg(ws.hist + (size_t)(b0 + i) * kE + e) : 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      tot += c[i];
      pre += b0 + i < blk ? c[i] : 0;
    }
  }
  s_pre[e] = pre;
  for (int i = threadIdx.x; i < 4 * kE; i += blockDim.x) (&mask[0][0])[i] = 0u;
  plan_groups(p, tot, G, ws, blk == 0);  // ends with a barrier
  const long long nb = gridDim.x;
  plan_units(G, ws.units_gu, false, (int)(G.n_gu * blk / nb), (int)(G.n_gu * (blk + 1) / nb),
             p.T);
  plan_units(G, ws.units_dn, true, (int)(G.n_dn * blk / nb), (int)(G.n_dn * (blk + 1) / nb),
             p.T);
  scatter_block(blk, p.T, topk_idx, perm, ws, mask, s_pre, G.off, G.poff, G.p_shared);
  pdl_trigger();
}

// The same for many token blocks, in two launches.  Plan (one block): thread e walks expert
// e's counts over the token blocks, storing each block's base (blkpre), then builds the group
// table, the global plan outputs and the whole unit lists.
__global__ void __launch_bounds__(256) route_plan_kernel(PlanArgs p, RouteWs ws) {
  __shared__ GroupTable G;
  pdl_wait();
  const int e = threadIdx.x;
  // loads first (read-only path), then the prefix stores: keeps 16 loads in flight
  int run = 0;
  for (int b0 = 0; b0 < p.nblk; b0 += 16) {
    int c[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      c[i] = b0 + i < p.nblk ? __ldg(ws.hist + (size_t)(b0 + i) * kE + e) : 0;
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if (b0 + i < p.nblk) {
        ws.blkpre[(size_t)(b0 + i) * kE + e] = run;
        run += c[i];
      }
  }
  plan_groups(p, run, G, ws, true);
  plan_units(G, ws.units_gu, false, 0, G.n_gu, p.T);
  plan_units(G, ws.units_dn, true, 0, G.n_dn, p.T);
  pdl_trigger();
}

// Scatter (one block of 128 threads per token block) from the plan's global outputs.
__global__ void __launch_bounds__(128) route_scatter_kernel(int T, const int32_t* topk_idx,
                                                            int32_t* perm, RouteWs ws) {
  __shared__ uint32_t mask[4][kE];
  __shared__ int s_pre[kE], s_off[kE], s_poff[kE + 1];
  pdl_wait();
  const int blk = blockIdx.x;
  for (int i = threadIdx.x; i < 4 * kE; i += blockDim.x) (&mask[0][0])[i] = 0u;
  for (int i = threadIdx.x; i < kE; i += blockDim.x) {
    s_pre[i] = __ldg(ws.blkpre + (size_t)blk * kE + i);
    s_off[i] = __ldg(ws.offsets + i);
    s_poff[i] = __ldg(ws.poff + i);
  }
  if (threadIdx.x == 0) s_poff[kE] = __ldg(ws.poff + kE);
  __syncthreads();
  scatter_block(blk, T, topk_idx, perm, ws, mask, s_pre, s_off, s_poff, s_poff[kE]);
  pdl_trigger();
}

}  // namespace

cudaError_t prepare_route_kernels() {
  return cudaFuncSetAttribute(router_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kRtSmem);
}

cudaError_t launch_router_topk(const CUtensorMap& tm_x, const CUtensorMap& tm_wr,
                               const float* bias, int T, const Dims& D, int32_t* topk_idx,
                               float* topk_w, const RouteWs& ws, cudaStream_t s) {
  RouterArgs a{bias, T, D.d, topk_idx, topk_w, ws.hist, ws.err};
  const int nblk = (T + kBlockTokens - 1) / kBlockTokens;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nblk * kRtCluster);
  cfg.blockDim = dim3(kRtThreads);
  cfg.dynamicSmemBytes = kRtSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kRtCluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, router_topk_kernel, tm_x, tm_wr, a);
}

cudaError_t launch_route_plan_scatter(int T, const Dims& D, const int32_t* topk_idx,
                                      int32_t* perm, const RouteWs& ws, cudaStream_t s) {
  const PlanArgs p = plan_args(T, D);
  const int nblk = p.nblk;
  if (nblk <= kFusedPlanBlocks)
    return launch_pdl(route_plan_scatter_kernel, dim3(nblk), dim3(256), 0, s, p, topk_idx, perm,
                      ws);
  cudaError_t e = launch_pdl(route_plan_kernel, dim3(1), dim3(256), 0, s, p, ws);
  if (e != cudaSuccess) return e;
  return launch_pdl(route_scatter_kernel, dim3(nblk), dim3(128), 0, s, T, topk_idx, perm, ws);
}

}  // namespace moe
