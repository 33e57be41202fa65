// Routing chain of the MoE layer on the GPU ("Optimizing on-device inference for Apple
// Silicon", § "Keep expert routing on the GPU"): router scores and top-8 selection, a
// histogram of assignments per expert, a prefix scan into start offsets, a scatter of the
// rows into their expert groups, and the block map (work units) of the grouped GEMMs.
// Nothing here waits for the host, and every result is deterministic: the histogram is
// kept per 128-token block and combined in block order, and ranks inside a block come
// from bit masks in token order, so no atomic ordering reaches an output.
#include "layer.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

// ---------------------------------------------------------------- router GEMM + top-8

// A cluster of four blocks per 128 tokens: block r computes the logits of experts
// [64r, 64r + 64) (tcgen05, M = 128 tokens, N = 64 experts, K = d).  The x tile is shared:
// each block loads a quarter of its rows and multicasts it to the four.  Each block keeps its
// 8 largest logits per token and writes them into the leader block's shared memory; the leader
// merges the 4 x 8 candidates, applies the softmax and counts the histogram.
constexpr int kRtCluster = 4;
constexpr int kRtN = kE / kRtCluster;                 // experts per block
constexpr int kRtStages = 6;
constexpr int kRtA = kBlockTokens * kBK * 2;          // x tile: 128 tokens x 64 (16 KB)
constexpr int kRtASlice = kRtA / kRtCluster;          // rows loaded (and multicast) per block
constexpr int kRtB = kRtN * kBK * 2;                  // router tile: 64 experts x 64 (8 KB)
constexpr int kRtStage = kRtA + kRtB;
constexpr int kRtThreads = 320;                       // producer, MMA, 8 epilogue warps
constexpr int kRtCand = kBlockTokens * kRtCluster * 8;  // leader: 4 lists of 8 per token
constexpr int kRtHalf = kBlockTokens * 2 * 8;           // each block: 2 half-lists per token
constexpr int kRtSmem = kRtStages * kRtStage + (kRtCand + kRtHalf) * 8 + 1024 + 2048;

struct RouterArgs {
  const float* bias;
  int T, d;
  int32_t* topk_idx;
  float* topk_w;
  int32_t* hist;
  int* err;
};

// Keeps the 8 largest (value, id) pairs in v/id, sorted by value descending; among equal
// values the earlier-inserted pair stays ahead (callers insert ids in ascending order).
__device__ __forceinline__ void top8_insert(float (&v)[8], int (&id)[8], float x, int e) {
  if (x > v[7]) {
    v[7] = x;
    id[7] = e;
#pragma unroll
    for (int i = 7; i > 0; --i) {
      if (v[i] > v[i - 1]) {
        float tv = v[i]; v[i] = v[i - 1]; v[i - 1] = tv;
        int ti = id[i]; id[i] = id[i - 1]; id[i - 1] = ti;
      }
    }
  }
}

// The 8 largest of L lists of 8 (each sorted by value descending, ids ascending among equal
// values; list l holding lower ids than list l + 1): eight steps, each taking the largest
// head, the lower list on equal values -- so ties still go to the lower id.
template <int L>
__device__ __forceinline__ void merge_top8(const float* cv, const int* ci, float (&v)[8],
                                           int (&id)[8]) {
  int pos[L];
#pragma unroll
  for (int l = 0; l < L; ++l) pos[l] = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    float bv = -INFINITY;
    int bl = 0;
#pragma unroll
    for (int l = 0; l < L; ++l) {
      const float hv = pos[l] < 8 ? cv[l * 8 + pos[l]] : -INFINITY;
      if (hv > bv) { bv = hv; bl = l; }
    }
    int bi = 0;
#pragma unroll
    for (int l = 0; l < L; ++l)
      if (l == bl) { bi = ci[l * 8 + pos[l]]; pos[l] += 1; }
    v[k] = bv;
    id[k] = bi;
  }
}

__global__ void __launch_bounds__(kRtThreads, 1)
    router_topk_kernel(const __grid_constant__ CUtensorMap tm_x,
                       const __grid_constant__ CUtensorMap tm_wr, RouterArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  float* cand_v = reinterpret_cast<float*>(smem + kRtStages * kRtStage);  // [128][4][8] leader
  int* cand_i = reinterpret_cast<int*>(cand_v + kRtCand);
  float* half_v = reinterpret_cast<float*>(cand_i + kRtCand);             // [128][2][8]
  int* half_i = reinterpret_cast<int*>(half_v + kRtHalf);
  uint64_t* full = reinterpret_cast<uint64_t*>(half_i + kRtHalf);
  uint64_t* empty = full + kRtStages;
  uint64_t* tfull = empty + kRtStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tfull + 1);
  int* hist_s = reinterpret_cast<int*>(tmem_slot + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int blk = (int)cluster_id_x();  // 128-token block
  const int KB = a.d / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRtStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kRtCluster);  // released by the MMA of every block of the cluster
    }
    mbar_init(tfull, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kRtN);
    tmem_relinquish();
  }
  for (int i = threadIdx.x; i < kE; i += blockDim.x) hist_s[i] = 0;
  tc_fence_before();
  cluster_sync();  // barriers of every block initialised before any multicast lands
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // x (and the bias) may come from the previous kernel on the stream

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tensormap(&tm_x);
      prefetch_tensormap(&tm_wr);
      const uint64_t keep = policy_evict_last();  // x and the router weights are re-read
      int stage = 0;
      uint32_t ph = 0;
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait(&empty[stage], ph ^ 1, a.err)) break;
        uint8_t* st = smem + stage * kRtStage;
        mbar_arrive_expect_tx(&full[stage], kRtStage);
        tma_load_2d_mc(st + rank * kRtASlice, &tm_x, &full[stage], kb * kBK,
                       blk * kBlockTokens + (int)rank * (kBlockTokens / kRtCluster),
                       (uint16_t)((1u << kRtCluster) - 1), keep);
        tma_load_2d(st + kRtA, &tm_wr, &full[stage], kb * kBK, (int)rank * kRtN, keep);
        if (++stage == kRtStages) { stage = 0; ph ^= 1; }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, kRtN);
      int stage = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait(&full[stage], ph, a.err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + stage * kRtStage), sb = sa + kRtA;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          mma_bf16(tmem, sdesc_k128(sa + kk * 32), sdesc_k128(sb + kk * 32), idesc,
                   (kb | kk) != 0);
        mma_commit_mc(&empty[stage], (uint16_t)((1u << kRtCluster) - 1));
        if (++stage == kRtStages) { stage = 0; ph ^= 1; }
      }
      if (ok) mma_commit(tfull);
    }
  } else {
    // epilogue: thread = one token row and one half (32) of this block's 64 experts
    const int q = warp & 3, half = (warp - 2) >> 2;
    const int m = q * 32 + lane;
    const bool have = mbar_wait(tfull, 0, a.err);
    tc_fence_after();
    float v[8];
    int id[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) { v[i] = -INFINITY; id[i] = 0; }
    if (have) {
#pragma unroll
      for (int c0 = 0; c0 < kRtN / 2; c0 += 16) {
        uint32_t r[16];
        tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(half * (kRtN / 2) + c0), r);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int e = (int)rank * kRtN + half * (kRtN / 2) + c0 + i;
          float x = __uint_as_float(r[i]);
          if (a.bias) x += __ldg(a.bias + e);
          top8_insert(v, id, x, e);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      half_v[(m * 2 + half) * 8 + j] = v[j];
      half_i[(m * 2 + half) * 8 + j] = id[j];
    }
    named_sync(1, 8 * 32);  // both halves of every token listed
    if (half == 0) {
      merge_top8<2>(half_v + m * 16, half_i + m * 16, v, id);
      const uint32_t dv = map_shared(cand_v + m * (kRtCluster * 8) + rank * 8, 0);
      const uint32_t di = map_shared(cand_i + m * (kRtCluster * 8) + rank * 8, 0);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        st_cluster_f32(dv + 4 * j, v[j]);
        st_cluster_s32(di + 4 * j, id[j]);
      }
    }
  }
  tc_fence_before();
  cluster_sync();  // candidates of all four blocks are in the leader's shared memory

  if (rank == 0 && warp >= 2 && ((warp - 2) >> 2) == 0) {
    const int q = warp & 3;
    const int m = q * 32 + lane;
    const int t = blk * kBlockTokens + m;
    float v[8];
    int id[8];
    merge_top8<kRtCluster>(cand_v + m * (kRtCluster * 8), cand_i + m * (kRtCluster * 8), v, id);
    // list the kept experts in ascending id
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
    float ex[8], s = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) { ex[j] = __expf(v[j] - mx); s += ex[j]; }
    if (t < a.T) {
      int4* pi = reinterpret_cast<int4*>(a.topk_idx + (size_t)t * kTopK);
      float4* pw = reinterpret_cast<float4*>(a.topk_w + (size_t)t * kTopK);
      pi[0] = make_int4(id[0], id[1], id[2], id[3]);
      pi[1] = make_int4(id[4], id[5], id[6], id[7]);
      pw[0] = make_float4(ex[0] / s, ex[1] / s, ex[2] / s, ex[3] / s);
      pw[1] = make_float4(ex[4] / s, ex[5] / s, ex[6] / s, ex[7] / s);
#pragma unroll
      for (int j = 0; j < 8; ++j) atomicAdd(&hist_s[id[j]], 1);
    }
    named_sync(2, 128);  // the four merging warps
    const int et = threadIdx.x - 64;
    a.hist[(size_t)blk * kE + et] = hist_s[et];
    a.hist[(size_t)blk * kE + et + 128] = hist_s[et + 128];
  }
  pdl_trigger();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kRtN);
}

// ---------------------------------------------------------------- plan

// Exclusive scans of N values over the 256 threads of the block: v[n] becomes the sum of v[n]
// over lower threads, total[n] the block sum.  Two barriers for all N scans.
template <int N>
__device__ __forceinline__ void block_scan_256(int (&v)[N], int* tmp, int (&total)[N]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x[N];
#pragma unroll
  for (int n = 0; n < N; ++n) {
    x[n] = v[n];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x[n], o);
      if (lane >= o) x[n] += y;
    }
    if (lane == 31) tmp[n * 8 + warp] = x[n];
  }
  __syncthreads();
#pragma unroll
  for (int n = 0; n < N; ++n) {
    int base = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const int c = tmp[n * 8 + w];
      base += w < warp ? c : 0;
      tot += c;
    }
    v[n] = base + x[n] - v[n];
    total[n] = tot;
  }
  __syncthreads();  // tmp may be reused
}

struct PlanArgs {
  int T, nblk, mt_f, mt_fs, mt_d;
};

// The expert groups of one plan, in shared memory: per expert the first gate/up and down unit,
// chunk count and size, padded start row, assignment count, first chunk id and offset; and the
// shared group's figures.
struct GroupTable {
  int gu0[kE], dn0[kE], nch[kE], cs[kE], poff[kE], cnt[kE], cid0[kE], off[kE];
  int tmp[8 * 5];
  int n_gu, n_dn, gu_s, dn_s, nch_s, cs_s, p_shared;
};

// Thread e (all 256 threads call it) with cnt = assignments to expert e: the exclusive scan into
// offsets, the padded group starts (groups start on 16-row boundaries; the shared expert's T rows
// follow the routed groups), and the unit bookkeeping: each group is cut into ceil(n / 192)
// nearly equal chunks of rows, and each chunk is paired with every weight row tile.  Routed
// units are listed by expert ascending; inside a group, weight tile major and chunk minor, so
// units that read the same weights are adjacent (the shared group's units are spread among
// them, see plan_units).  The writer block also stores the
// global offsets, group starts and unit counts, zeroes the schedule counter, the chunk counters
// and the grow entries of padding rows.
__device__ void plan_groups(const PlanArgs& p, int cnt, GroupTable& G, const RouteWs& ws,
                            bool writer) {
  const int e = threadIdx.x;
  const int pc = round_up(cnt, kRowAlign);
  const int nch = (cnt + kChunkRows - 1) / kChunkRows;
  int v[5] = {cnt, pc, nch * p.mt_f, nch * p.mt_d, nch};
  int tot[5];
  block_scan_256<5>(v, G.tmp, tot);
  const int nch_s = (p.T + kChunkRows - 1) / kChunkRows;
  const int cs_s = nch_s ? round_up((p.T + nch_s - 1) / nch_s, kRowAlign) : 0;
  const int gu_s = nch_s * p.mt_fs, dn_s = nch_s * p.mt_d;
  const int p_shared = tot[1];
  const int cid0 = nch_s + v[4];
  G.gu0[e] = gu_s + v[2];
  G.dn0[e] = dn_s + v[3];
  G.nch[e] = nch;
  G.cs[e] = nch ? round_up((cnt + nch - 1) / nch, kRowAlign) : 0;
  G.poff[e] = v[1];
  G.cnt[e] = cnt;
  G.cid0[e] = cid0;
  G.off[e] = v[0];
  if (e == 0) {
    G.n_gu = gu_s + tot[2];
    G.n_dn = dn_s + tot[3];
    G.gu_s = gu_s;
    G.dn_s = dn_s;
    G.nch_s = nch_s;
    G.cs_s = cs_s;
    G.p_shared = p_shared;
  }
  if (writer) {
    ws.offsets[e] = v[0];
    ws.poff[e] = v[1];
    if (e == kE - 1) {
      ws.offsets[kE] = tot[0];
      ws.poff[kE] = p_shared;
      ws.poff[kE + 1] = p_shared + round_up(p.T, kRowAlign);
      ws.n_units[0] = gu_s + tot[2];
      ws.n_units[1] = dn_s + tot[3];
      *ws.next_unit = 0;
    }
    for (int r = v[1] + cnt; r < v[1] + pc; ++r) ws.grow[r] = 0;
    if (e == 0)
      for (int r = p_shared + p.T; r < p_shared + round_up(p.T, kRowAlign); ++r) ws.grow[r] = 0;
    for (int c = 0; c < nch; ++c) ws.chunk_done[cid0 + c] = 0;
    for (int c = threadIdx.x; c < nch_s; c += blockDim.x) ws.chunk_done[c] = 0;
  }
  __syncthreads();
}

// Last index e in [0, kE) with start[e] <= u (start is non-decreasing); the group holding unit u.
__device__ __forceinline__ int find_group(const int* start, int u) {
  int lo = 0, hi = kE - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (start[mid] <= u) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Writes units [lo, hi) of one list (gate/up: dn = false) from the group table: consecutive
// threads, consecutive units.  The shared group's units (chunk major, weight tile minor) are
// spread evenly through the list -- position u holds a shared unit when the count
// floor((u + 1) s / n) of shared units up to u grows there -- so that at every point of the
// schedule most blocks stream routed weights from HBM while a few run the shared expert,
// whose weights stay in L2; the routed units keep their order (group of a routed unit found by
// binary search over the group starts).
__device__ void plan_units(const GroupTable& G, Unit* units, bool dn, int lo, int hi, int T) {
  const int* start = dn ? G.dn0 : G.gu0;
  const long long n = dn ? G.n_dn : G.n_gu;
  const int ns = dn ? G.dn_s : G.gu_s;
  const int mts = G.nch_s ? ns / G.nch_s : 1;  // weight tiles per shared chunk
  for (int u = lo + (int)threadIdx.x; u < hi; u += blockDim.x) {
    const int upto = (int)(((long long)u + 1) * ns / n), before = (int)((long long)u * ns / n);
    if (upto > before) {
      const int c = before / mts, mt = before % mts;
      units[u] = Unit{kE, G.p_shared + c * G.cs_s, min(G.cs_s, T - c * G.cs_s), mt, c};
    } else {
      const int v = u - upto + ns;  // position in the list with the shared units first
      const int g = find_group(start, v), l = v - start[g], nc = G.nch[g];
      const int mt = l / nc, c = l % nc, cs = G.cs[g];
      units[u] = Unit{g, G.poff[g] + c * cs, min(cs, G.cnt[g] - c * cs), mt, G.cid0[g] + c};
    }
  }
}

// Scatter of the tokens of token block `blk` (threads 0..127, one token each, four warps of
// 32): the rank of (t, e) among the assignments to expert e = `pre[e]` (assignments of earlier
// blocks) + those of earlier warps of this block + those of lower lanes of this warp, counted
// from per-warp bit masks of the tokens that chose e.  mask must be zero on entry; every thread
// of the block calls this (it holds one barrier).
__device__ __forceinline__ void scatter_block(int blk, int T, const int32_t* topk_idx,
                                              int32_t* perm, const RouteWs& ws,
                                              uint32_t (*mask)[kE], const int* pre,
                                              const int* off, const int* poff, int p_shared) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blk * kBlockTokens + (int)threadIdx.x;
  const bool valid = threadIdx.x < kBlockTokens && t < T;
  int e[8];
  if (valid) {
    const int4* pi = reinterpret_cast<const int4*>(topk_idx + (size_t)t * kTopK);
    const int4 a = pi[0], b = pi[1];
    e[0] = a.x; e[1] = a.y; e[2] = a.z; e[3] = a.w;
    e[4] = b.x; e[5] = b.y; e[6] = b.z; e[7] = b.w;
#pragma unroll
    for (int j = 0; j < 8; ++j) atomicOr(&mask[warp][e[j]], 1u << lane);
  }
  __syncthreads();
  if (valid) {
    const uint32_t below = (1u << lane) - 1u;
    int pr[9];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int ee = e[j];
      int rank = pre[ee] + __popc(mask[warp][ee] & below);
      for (int w = 0; w < warp; ++w) rank += __popc(mask[w][ee]);
      perm[off[ee] + rank] = t * kTopK + j;
      pr[j] = poff[ee] + rank;
      ws.grow[pr[j]] = t;
    }
    pr[8] = p_shared + t;
    ws.grow[pr[8]] = t;
    int* prow = ws.prow + (size_t)t * 9;
#pragma unroll
    for (int j = 0; j < 9; ++j) prow[j] = pr[j];
  }
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
  // down units cover 256 outputs (two 128-row weight tiles; the last may have one)
  const int nblk = (T + kBlockTokens - 1) / kBlockTokens;
  PlanArgs p{T, nblk, D.f / kMTile, D.fs / kMTile, (D.d + 2 * kMTile - 1) / (2 * kMTile)};
  if (nblk <= kFusedPlanBlocks)
    return launch_pdl(route_plan_scatter_kernel, dim3(nblk), dim3(256), 0, s, p, topk_idx, perm,
                      ws);
  cudaError_t e = launch_pdl(route_plan_kernel, dim3(1), dim3(256), 0, s, p, ws);
  if (e != cudaSuccess) return e;
  return launch_pdl(route_scatter_kernel, dim3(nblk), dim3(128), 0, s, T, topk_idx, perm, ws);
}

}  // namespace moe
