// Grouped expert GEMMs on the 5th-generation tensor cores and the weighted combine.
//
// "Optimizing on-device inference for Apple Silicon": the grouped GEMM needs the rows routed
// to each expert stored together (§ "Keep expert routing on the GPU"), its tile follows the
// expert's load (§ "Match tile size to expert load"), it accumulates in fp32 and writes bf16
// (§ "Dequantize weights during matrix multiplication"), and the gated activation is fused
// into the input projections (§ "Reduce intermediate and state traffic").
//
// GB300 design: the weights take the MMA's M = 128 side and the routed token rows the
// N side (16..256 in steps of 16), so an expert with few tokens still uses full-height MMAs
// and its weight tile is read once per chunk of up to 256 tokens.  One persistent block per
// SM walks the work-unit list: the weight tiles reach a shared-memory ring by TMA (128-row
// tiles) and the routed token rows by 16-byte cp.async gathers straight from x (so
// no permuted copy of x is ever written), warp 1 issues tcgen05.mma into TMEM, and the
// epilogue warps drain TMEM (SwiGLU for gate/up, plain bf16 for down) while the ring refills.
#include "layer.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kTileA = kMTile * kBK * 2;     // 128 weight rows x 64 (16 KB)
constexpr int kTileB = kChunkRows * kBK * 2; // up to 256 token rows x 64 (32 KB)

// ---------------------------------------------------------------- gate/up + SwiGLU

constexpr int kGuStages = 3;
constexpr int kGuStage = 2 * kTileA + kTileB;  // gate tile | up tile | token rows
constexpr int kGuSmem = kGuStages * kGuStage + 1024 + 1024;
constexpr int kGuThreads = 384;                // 12 warps, roles below
constexpr int kGuRowThreads = 64;              // warps 2-3: token-row copies
constexpr int kGuEpiWarps = 8;                 // warps 4-11: two per TMEM lane quadrant

struct GuArgs {
  const Unit* units;
  const int32_t* n_units;
  const int32_t* grow;
  const __nv_bfloat16* x;
  __nv_bfloat16* h;
  int d, f, hdim;
  int* err;
};

// Warp roles: 0 = TMA producer of the gate and up weight tiles; 1 = MMA issuer (and TMEM
// owner); 2-3 = producers of the token rows (gathered from x by 16-byte cp.async straight
// into the 128-byte-swizzled layout: row r, chunk c lands at r*128 + ((c ^ (r & 7)) * 16));
// 4-11 = epilogue, two warps per TMEM lane quadrant, each taking alternate 16-column chunks.
__global__ void __launch_bounds__(kGuThreads, 1)
    gateup_kernel(const __grid_constant__ CUtensorMap tm_wg, const __grid_constant__ CUtensorMap tm_wu,
                  const __grid_constant__ CUtensorMap tm_wsg,
                  const __grid_constant__ CUtensorMap tm_wsu, GuArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kGuStages * kGuStage);
  uint64_t* empty = full + kGuStages;
  uint64_t* tfull = empty + kGuStages;
  uint64_t* tempty = tfull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KB = a.d / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGuStages; ++s) {
      mbar_init(&full[s], 1 + kGuRowThreads);  // weight TMA + one arrival per row thread
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, kGuEpiWarps);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();
  const int n_units = *a.n_units;

  if (warp == 0) {
    // ---- weight tiles (gate and up, 128 rows x 64 each) by tiled TMA
    if (lane == 0) {
      prefetch_tensormap(&tm_wg);
      prefetch_tensormap(&tm_wu);
      prefetch_tensormap(&tm_wsg);
      prefetch_tensormap(&tm_wsu);
      const uint64_t stream_w = policy_evict_first();  // each weight tile is read once
      int stage = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        const Unit U = a.units[u];
        const bool shared = U.g == kE;
        const CUtensorMap* mg = shared ? &tm_wsg : &tm_wg;
        const CUtensorMap* mu = shared ? &tm_wsu : &tm_wu;
        const int arow = (shared ? 0 : U.g * a.f) + U.mt * kMTile;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&empty[stage], ph ^ 1, a.err)) { ok = false; break; }
          uint8_t* st = smem + stage * kGuStage;
          mbar_arrive_expect_tx(&full[stage], 2 * kTileA);
          tma_load_2d(st, mg, &full[stage], kb * kBK, arow, stream_w);
          tma_load_2d(st + kTileA, mu, &full[stage], kb * kBK, arow, stream_w);
          if (++stage == kGuStages) { stage = 0; ph ^= 1; }
        }
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer: gate accumulator in TMEM columns [0, N), up in [256, 256 + N)
    if (lane == 0) {
      int stage = 0;
      uint32_t ph = 0, tph = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        const Unit U = a.units[u];
        const int N = round_up(U.nrows, kRowAlign);
        const uint32_t idesc = idesc_bf16(128, N);
        if (!mbar_wait(tempty, tph ^ 1, a.err)) break;
        tc_fence_after();
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&full[stage], ph, a.err)) { ok = false; break; }
          fence_proxy_async_smem();  // token rows were written by cp.async (generic proxy)
          tc_fence_after();
          const uint32_t sg = smem_u32(smem + stage * kGuStage);
          const uint32_t su = sg + kTileA, sb = sg + 2 * kTileA;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t bd = sdesc_k128(sb + kk * 32);
            const uint32_t acc = (kb | kk) != 0;
            mma_bf16(tmem, sdesc_k128(sg + kk * 32), bd, idesc, acc);
            mma_bf16(tmem + 256, sdesc_k128(su + kk * 32), bd, idesc, acc);
          }
          mma_commit(&empty[stage]);
          if (++stage == kGuStages) { stage = 0; ph ^= 1; }
        }
        if (ok) mma_commit(tfull);
        tph ^= 1;
      }
    }
  } else if (warp < 4) {
    // ---- token rows: thread (crow, chunk) copies 16-byte chunk `chunk` of rows crow + 8i
    const int bt = threadIdx.x - 64;
    const int crow = bt >> 3, chunk = bt & 7;
    const uint32_t swz = (uint32_t)((chunk ^ crow) << 4);  // (r & 7) == crow for every row
    const uint64_t keep_x = policy_evict_last();            // x rows are gathered many times
    int stage = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const Unit U = a.units[u];
      const int N = round_up(U.nrows, kRowAlign);
      const int nr = N / 8;  // rows per thread, <= 32
      const __nv_bfloat16* src[kChunkRows / 8];
#pragma unroll
      for (int i = 0; i < kChunkRows / 8; ++i)
        src[i] = a.x + (size_t)(i < nr ? __ldg(a.grow + U.p0 + crow + 8 * i) : 0) * a.d +
                 chunk * 8;
      for (int kb = 0; kb < KB; ++kb) {
        const bool w = mbar_wait(&empty[stage], ph ^ 1, a.err);
        if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
        const uint32_t sb = smem_u32(smem + stage * kGuStage + 2 * kTileA) + crow * 128 + swz;
#pragma unroll
        for (int i = 0; i < kChunkRows / 8; ++i)
          if (i < nr) cp_async_16(sb + i * 1024, src[i] + kb * kBK, keep_x);
        cp_async_arrive_noinc(&full[stage]);
        if (++stage == kGuStages) { stage = 0; ph ^= 1; }
      }
    }
  } else {
    // ---- epilogue: thread = one feature row; h = silu(gate) * up for each token column
    const int q = warp & 3, half = (warp - 4) >> 2;
    const int m = q * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    uint32_t tph = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      const Unit U = a.units[u];
      const int N = round_up(U.nrows, kRowAlign);
      const bool w = mbar_wait(tfull, tph, a.err);
      if (!__all_sync(0xffffffffu, w)) break;
      tc_fence_after();
      __nv_bfloat16* hp = a.h + (size_t)U.p0 * a.hdim + U.mt * kMTile + m;
      for (int j0 = half * 16; j0 < N; j0 += 32) {
        uint32_t g[16], v[16];
        tmem_ld16(tmem + lane_off + (uint32_t)j0, g);
        tmem_ld16(tmem + lane_off + 256u + (uint32_t)j0, v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i)
          hp[(size_t)(j0 + i) * a.hdim] =
              __float2bfloat16_rn(silu_mul(__uint_as_float(g[i]), __uint_as_float(v[i])));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty);
      tph ^= 1;
    }
  }
  pdl_trigger();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------- down

constexpr int kDnStages = 4;
constexpr int kDnStage = kTileA + kTileB;
constexpr int kDnSmem = kDnStages * kDnStage + 1024 + 1024;

struct DnArgs {
  const Unit* units;
  const int32_t* n_units;
  __nv_bfloat16* ys;
  int d, f, fs;
  int* err;
};

__global__ void __launch_bounds__(192, 1)
    down_kernel(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_wd,
                const __grid_constant__ CUtensorMap tm_wsd, DnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kDnStages * kDnStage);
  uint64_t* empty = full + kDnStages;
  uint64_t* tfull = empty + kDnStages;  // [2]
  uint64_t* tempty = tfull + 2;         // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kDnStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 4);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();
  const int n_units = *a.n_units;

  if (warp == 0) {
    // ---- producer: weight tile + 16-row tiles of h
    if (lane == 0) {
      prefetch_tensormap(&tm_h);
      prefetch_tensormap(&tm_wd);
      prefetch_tensormap(&tm_wsd);
    }
    const uint64_t stream_w = policy_evict_first();
    const uint64_t keep_h = policy_evict_last();
    int stage = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const Unit U = a.units[u];
      const int N = round_up(U.nrows, kRowAlign);
      const bool shared = U.g == kE;
      const int K = shared ? a.fs : a.f;
      const CUtensorMap* mw = shared ? &tm_wsd : &tm_wd;
      const int arow = (shared ? 0 : U.g * a.d) + U.mt * kMTile;
      const uint32_t bytes = kTileA + (uint32_t)N * kBK * 2;
      for (int kb = 0; kb < K / kBK; ++kb) {
        const bool w = mbar_wait(&empty[stage], ph ^ 1, a.err);
        if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
        uint8_t* st = smem + stage * kDnStage;
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[stage], bytes);
          tma_load_2d(st, mw, &full[stage], kb * kBK, arow, stream_w);
        }
        __syncwarp();
        if (lane < N / 16)
          tma_load_2d(st + kTileA + lane * 2048, &tm_h, &full[stage], kb * kBK, U.p0 + 16 * lane,
                      keep_h);
        if (++stage == kDnStages) { stage = 0; ph ^= 1; }
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer: two accumulator slots of 256 columns, alternating per unit
    if (lane == 0) {
      int stage = 0, slot = 0;
      uint32_t ph = 0, tph[2] = {0, 0};
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        const Unit U = a.units[u];
        const int N = round_up(U.nrows, kRowAlign);
        const int K = U.g == kE ? a.fs : a.f;
        const uint32_t idesc = idesc_bf16(128, N);
        const uint32_t acc_col = tmem + 256u * slot;
        if (!mbar_wait(&tempty[slot], tph[slot] ^ 1, a.err)) break;
        tc_fence_after();
        for (int kb = 0; kb < K / kBK; ++kb) {
          if (!mbar_wait(&full[stage], ph, a.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * kDnStage), sb = sa + kTileA;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            mma_bf16(acc_col, sdesc_k128(sa + kk * 32), sdesc_k128(sb + kk * 32), idesc,
                     (kb | kk) != 0);
          mma_commit(&empty[stage]);
          if (++stage == kDnStages) { stage = 0; ph ^= 1; }
        }
        if (ok) mma_commit(&tfull[slot]);
        tph[slot] ^= 1;
        slot ^= 1;
      }
    }
  } else {
    // ---- epilogue: thread = one output feature; ys[row][n] = bf16(acc)
    const int q = warp & 3;
    const int m = q * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    uint32_t tph[2] = {0, 0};
    int slot = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      const Unit U = a.units[u];
      const int N = round_up(U.nrows, kRowAlign);
      const bool w = mbar_wait(&tfull[slot], tph[slot], a.err);
      if (!__all_sync(0xffffffffu, w)) break;
      tc_fence_after();
      __nv_bfloat16* yp = a.ys + (size_t)U.p0 * a.d + U.mt * kMTile + m;
      for (int j0 = 0; j0 < N; j0 += 16) {
        uint32_t r[16];
        tmem_ld16(tmem + lane_off + 256u * slot + (uint32_t)j0, r);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i)
          yp[(size_t)(j0 + i) * a.d] = __float2bfloat16_rn(__uint_as_float(r[i]));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[slot]);
      tph[slot] ^= 1;
      slot ^= 1;
    }
  }
  pdl_trigger();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------- combine

// One block per token, one thread per 8 consecutive outputs (16-byte loads of ys rows).
// acc = sum over j = 0..7 (ascending expert id) of w_j * ys[row_j], then + ys[shared row],
// in fp32, rounded once to bf16.
__global__ void __launch_bounds__(256) combine_kernel(int d, const float* topk_w,
                                                      const int32_t* prow,
                                                      const __nv_bfloat16* ys,
                                                      __nv_bfloat16* y) {
  pdl_wait();
  const int t = blockIdx.x;
  float w[8];
  int r[9];
#pragma unroll
  for (int j = 0; j < 8; ++j) w[j] = topk_w[(size_t)t * kTopK + j];
#pragma unroll
  for (int j = 0; j < 9; ++j) r[j] = prow[(size_t)t * 9 + j];
  for (int c = threadIdx.x; c < d / 8; c += blockDim.x) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
    for (int j = 0; j < 9; ++j) {
      const uint4 v = *reinterpret_cast<const uint4*>(ys + (size_t)r[j] * d + c * 8);
      const float wj = j < 8 ? w[j] : 1.0f;
      const uint32_t p[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] += wj * bf16_lo(p[i]);
        acc[2 * i + 1] += wj * bf16_hi(p[i]);
      }
    }
    uint4 o;
    uint32_t* po = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
      po[i] = *reinterpret_cast<uint32_t*>(&b2);
    }
    *reinterpret_cast<uint4*>(y + (size_t)t * d + c * 8) = o;
  }
  pdl_trigger();
}

}  // namespace

cudaError_t prepare_expert_kernels() {
  cudaError_t e = cudaFuncSetAttribute(gateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kGuSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDnSmem);
}

cudaError_t launch_gateup(const __nv_bfloat16* x, const CUtensorMap& tm_wg,
                          const CUtensorMap& tm_wu, const CUtensorMap& tm_wsg,
                          const CUtensorMap& tm_wsu, const Dims& D, const RouteWs& ws,
                          __nv_bfloat16* h, int grid, cudaStream_t s) {
  GuArgs a{ws.units_gu, ws.n_units, ws.grow, x, h, D.d, D.f, D.hdim, ws.err};
  return launch_pdl(gateup_kernel, dim3(grid), dim3(kGuThreads), kGuSmem, s, tm_wg, tm_wu, tm_wsg,
                    tm_wsu, a);
}

cudaError_t launch_down(const CUtensorMap& tm_h, const CUtensorMap& tm_wd,
                        const CUtensorMap& tm_wsd, const Dims& D, const RouteWs& ws,
                        __nv_bfloat16* ys, int grid, cudaStream_t s) {
  DnArgs a{ws.units_dn, ws.n_units + 1, ys, D.d, D.f, D.fs, ws.err};
  return launch_pdl(down_kernel, dim3(grid), dim3(192), kDnSmem, s, tm_h, tm_wd, tm_wsd, a);
}

cudaError_t launch_combine(int T, const Dims& D, const float* topk_w, const RouteWs& ws,
                           const __nv_bfloat16* ys, __nv_bfloat16* y, cudaStream_t s) {
  return launch_pdl(combine_kernel, dim3(T), dim3(256), 0, s, D.d, topk_w,
                    (const int32_t*)ws.prow, ys, y);
}

}  // namespace moe
