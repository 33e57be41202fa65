// The plan of the grouped GEMMs from the routing (used by the routing kernels and by the
// small-call router's last block): exclusive scans of the per-expert counts into offsets and
// padded group starts, the work-unit lists, and the scatter of a block of tokens into their
// expert groups.  "Optimizing on-device inference for Apple Silicon", § "Keep expert routing
// on the GPU": histogram, prefix scan, scatter and block map stay on the GPU.
#pragma once

#include "layer.cuh"

namespace moe {
namespace {

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

// The plan of T tokens: 128-token blocks; weight tiles per gate/up unit of a routed and of the
// shared group, and per down unit (256 outputs: two 128-row weight tiles, the last may have one).
inline PlanArgs plan_args(int T, const Dims& D) {
  return PlanArgs{T, (T + kBlockTokens - 1) / kBlockTokens, D.f / kMTile, D.fs / kMTile,
                  (D.d + 2 * kMTile - 1) / (2 * kMTile)};
}

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

}  // namespace
}  // namespace moe
