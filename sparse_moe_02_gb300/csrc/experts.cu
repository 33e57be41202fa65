// Grouped expert GEMMs on the 5th-generation tensor cores and the weighted combine.
//
// "Optimizing on-device inference for Apple Silicon": the grouped GEMM needs the rows routed
// to each expert stored together (§ "Keep expert routing on the GPU"), its tile follows the
// expert's load (§ "Match tile size to expert load"), it accumulates in fp32 and writes bf16
// (§ "Dequantize weights during matrix multiplication"), and the gated activation is fused
// into the input projections (§ "Reduce intermediate and state traffic").
//
// GB300 design: the weights take the MMA's M = 128 side and the routed token rows the
// N side (16..192 in steps of 16), so an expert with few tokens still uses full-height MMAs
// and its weight tile is read once per chunk of up to 192 tokens.  One persistent block per
// SM walks the work-unit list: the weight tiles reach a shared-memory ring by TMA (128-row
// tiles) and the routed token rows by 16-byte cp.async gathers straight from x (so
// no permuted copy of x is ever written), warp 1 issues tcgen05.mma into TMEM, and the
// epilogue warps drain TMEM (SwiGLU for gate/up, plain bf16 for down) while the ring refills.
#include "layer.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kTileA = kMTile * kBK * 2;     // 128 weight rows x 64 (16 KB)
constexpr int kTileB = kChunkRows * kBK * 2; // up to 192 token rows x 64 (24 KB)
static_assert((kChunkRows + kHBoxRows - 1) / kHBoxRows * kHBoxRows <= kChunkRows,
              "the h boxes of a down unit fit its token-row tile");

// ---------------------------------------------------------------- gate/up + down, one launch

// Ring of pipeline stages.  bf16 weights: 4 stages of (weight tile(s) | token rows).  4-bit
// weights: 6 stages of (the two tiles' codes, 128 rows x 32 bytes each | token rows); the
// dequantizing warps turn a stage's codes into bf16 tiles in tensor memory, from where the
// MMA reads its A operand.
template <bool Q4>
struct XCfg {
  static constexpr int kStages = Q4 ? 6 : 4;
  static constexpr int kBOff = Q4 ? 2 * kMTile * (kBK / 2) : 2 * kTileA;  // token rows
  static constexpr int kStage = kBOff + kTileB;
  static constexpr int kSmem = kStages * kStage + 1024 + 1024;
  static constexpr int kDqWarps = Q4 ? 8 : 0;                 // warps 12-19 (4-bit only)
  static constexpr int kThreads = 384 + 32 * kDqWarps;
};
constexpr int kXRowThreads = 64;               // warps 2-3: token-row copies (gate/up units)
constexpr int kXEpiWarps = 8;                  // warps 4-11: two per TMEM lane quadrant
constexpr int kXQueue = 4;                     // unit indices handed out ahead
constexpr int kQTile = kMTile * (kBK / 2);     // one stage's codes of one 128-row tile (4 KB)
// TMEM columns: accumulators [0, N) and [256, 256 + N) with N <= 192; the 4-bit path's two
// dequantized A buffers (two 32-column tiles each) sit in the columns above them
__device__ __forceinline__ uint32_t abuf_col(int b) { return b ? 448u : 192u; }

// 4-bit scales and biases of the six expert matrices (gate, up, down, shared gate, shared up,
// shared down): group (r, kb) of a matrix with K inputs per row at r * (K / 64) + kb
struct XQ4 {
  const __nv_bfloat16* s[6];
  const __nv_bfloat16* b[6];
};

struct XArgs {
  const Unit* units_gu;
  const Unit* units_dn;
  const int32_t* n_units;  // [2]: gate/up, down
  int32_t* next_unit;      // dynamic schedule: next unit index to hand out (zeroed by the plan)
  int32_t* chunk_done;
  const int32_t* grow;
  const __nv_bfloat16* x;
  __nv_bfloat16* h;
  __nv_bfloat16* ys;
  int d, f, fs, hdim;
  int* err;
  XQ4 q4;
};

struct XUnit {
  Unit u;
  bool down;
};

// Eight 4-bit codes (one 32-bit word: input 2i in the lower nibble of byte i) to four bf16
// pairs scale * q + bias, input 2i in the low half of pair i.  0x4300 | q is the bf16 value
// 128 + q exactly, so (128 + q) - 128 is q exactly, and the fused multiply-add rounds
// scale * q + bias once to bf16.
__device__ __forceinline__ void dequant_q4x8(uint32_t c, uint32_t s2, uint32_t b2, uint32_t* o) {
  const uint32_t lo = c & 0x0F0F0F0Fu;         // inputs 0, 2, 4, 6
  const uint32_t hi = (c >> 4) & 0x0F0F0F0Fu;  // inputs 1, 3, 5, 7
  const uint32_t p0 = __byte_perm(lo, hi, 0x5140);  // bytes: inputs 0 1 2 3
  const uint32_t p1 = __byte_perm(lo, hi, 0x7362);  // inputs 4 5 6 7
  const uint32_t m[4] = {__byte_perm(p0, 0x43434343u, 0x4140), __byte_perm(p0, 0x43434343u, 0x4342),
                         __byte_perm(p1, 0x43434343u, 0x4140), __byte_perm(p1, 0x43434343u, 0x4342)};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t qv;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(qv) : "r"(m[i]), "r"(0x3F803F80u), "r"(0xC300C300u));
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(o[i]) : "r"(qv), "r"(s2), "r"(b2));
  }
}

// One row's 64 codes of a step (two 16-byte words in shared memory) to 32 columns of bf16
// pairs with scale s and bias b (bf16 bits).
__device__ __forceinline__ void dequant_q4_row(const uint4* cp, uint32_t s, uint32_t b,
                                               uint32_t* v) {
  const uint4 c0 = cp[0], c1 = cp[1];
  const uint32_t s2 = s | (s << 16), b2 = b | (b << 16);
  dequant_q4x8(c0.x, s2, b2, v + 0);
  dequant_q4x8(c0.y, s2, b2, v + 4);
  dequant_q4x8(c0.z, s2, b2, v + 8);
  dequant_q4x8(c0.w, s2, b2, v + 12);
  dequant_q4x8(c1.x, s2, b2, v + 16);
  dequant_q4x8(c1.y, s2, b2, v + 20);
  dequant_q4x8(c1.z, s2, b2, v + 24);
  dequant_q4x8(c1.w, s2, b2, v + 28);
}

__device__ __forceinline__ XUnit unit_at(const XArgs& a, int i, int n_gu) {
  XUnit r;
  r.down = i >= n_gu;
  r.u = r.down ? a.units_dn[i - n_gu] : a.units_gu[i];
  return r;
}

// One persistent block per SM walks a combined list: every gate/up unit, then every down unit,
// handed out in list order by an atomic counter (the TMA producer lane takes the next index and
// passes it to the other roles through a small shared-memory queue).  Gate/up unit: 128 features of one group against up to
// 192 token rows; gate and up accumulators fill TMEM columns [0, N) and [256, 256 + N) (both
// halves); epilogue h = silu(gate) * up -> bf16, then the unit's chunk counter is incremented.
// Down unit: 256 outputs of one group as two 128-row weight tiles sharing the h rows, the two
// accumulators in the two TMEM halves; its producer waits for the chunk's counter to reach the
// number of gate/up tiles before loading h rows.
// Warp roles: 0 = TMA producer (weight tiles; h rows of down units); 1 = MMA issuer (TMEM
// owner); 2-3 = token-row producers of gate/up units (16-byte cp.async gathers from x into
// the 128-byte swizzle; for down units they only arrive); 4-11 = epilogue; with 4-bit weights
// 12-19 = dequantization (two groups of four warps on alternate steps).
// 4-bit weights (§ "Dequantize weights during matrix multiplication"): the weight maps are
// maps of the code bytes (box 32 bytes x 128 rows, no swizzle), each group's scale and bias
// come from a.q4, and the MMA takes A from tensor memory instead of shared memory.
template <bool Q4>
__global__ void __launch_bounds__(XCfg<Q4>::kThreads, 1)
    experts_kernel(const __grid_constant__ CUtensorMap tm_wg,
                   const __grid_constant__ CUtensorMap tm_wu,
                   const __grid_constant__ CUtensorMap tm_wsg,
                   const __grid_constant__ CUtensorMap tm_wsu,
                   const __grid_constant__ CUtensorMap tm_h,
                   const __grid_constant__ CUtensorMap tm_wd,
                   const __grid_constant__ CUtensorMap tm_wsd, XArgs a) {
  using C = XCfg<Q4>;
  constexpr int kXStages = C::kStages;
  constexpr int kXStage = C::kStage;
  constexpr int kXQueueReaders = 2 + 1 + kXEpiWarps + C::kDqWarps;  // every warp but the TMA's
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kXStages * kXStage);
  uint64_t* empty = full + kXStages;
  uint64_t* cfull = empty + kXStages;  // [kXStages] codes landed (4-bit)
  uint64_t* aempty = cfull + kXStages; // [2] dequantized A buffer free again (4-bit)
  uint64_t* tfull = aempty + 2;        // [2] TMEM halves
  uint64_t* tempty = tfull + 2;        // [2]
  uint64_t* qfull = tempty + 2;        // [kXQueue] unit-index queue
  uint64_t* qempty = qfull + kXQueue;  // [kXQueue]
  int* qidx = reinterpret_cast<int*>(qempty + kXQueue);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(qidx + kXQueue);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kXStages; ++s) {
      // TMA producer + one arrival per row thread (+ one per warp of a dequantizing group)
      mbar_init(&full[s], 1 + kXRowThreads + C::kDqWarps / 2);
      mbar_init(&empty[s], 1);
      mbar_init(&cfull[s], 1);
    }
    mbar_init(&aempty[0], 1);
    mbar_init(&aempty[1], 1);
    for (int i = 0; i < kXQueue; ++i) {
      mbar_init(&qfull[i], 1);
      mbar_init(&qempty[i], kXQueueReaders);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], kXEpiWarps);
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
  const int n_gu = a.n_units[0];
  const int n_all = n_gu + a.n_units[1];
  // reader side of the unit queue: the k-th unit this block processes (-1: no more units);
  // one arrival per reading warp releases the slot
  auto next_unit = [&](int k, bool& ok) {
    const int q = k % kXQueue;
    const bool w = mbar_wait(&qfull[q], (k / kXQueue) & 1, a.err);
    ok = __all_sync(0xffffffffu, w);
    const int i = ok ? *reinterpret_cast<volatile int*>(&qidx[q]) : -1;
    __syncwarp();
    if (lane == 0) mbar_arrive(&qempty[q]);
    return i;
  };
  // the same for a role that runs on a single lane (the MMA issuer)
  auto next_unit_1 = [&](int k, bool& ok) {
    const int q = k % kXQueue;
    ok = mbar_wait(&qfull[q], (k / kXQueue) & 1, a.err);
    const int i = ok ? *reinterpret_cast<volatile int*>(&qidx[q]) : -1;
    mbar_arrive(&qempty[q]);
    return i;
  };

  if (warp == 0) {
    // ---- TMA producer
    if (lane == 0) {
      prefetch_tensormap(&tm_wg);
      prefetch_tensormap(&tm_wu);
      prefetch_tensormap(&tm_wsg);
      prefetch_tensormap(&tm_wsu);
      prefetch_tensormap(&tm_h);
      prefetch_tensormap(&tm_wd);
      prefetch_tensormap(&tm_wsd);
      const uint64_t stream_w = policy_evict_first();  // a routed weight tile is read once
      const uint64_t keep_h = policy_evict_last();     // h rows; the shared expert's weights
      int stage = 0;
      uint32_t ph = 0;
      bool ok = true;
      // queue writer: index k goes to slot k % kXQueue once its previous use is read by all
      int kq = 0;
      auto push = [&](int i) {
        const int q = kq % kXQueue;
        if (kq >= kXQueue && !mbar_wait(&qempty[q], ((kq / kXQueue) - 1) & 1, a.err)) return false;
        qidx[q] = i;
        mbar_arrive(&qfull[q]);
        ++kq;
        return true;
      };
      int cur = atomicAdd(a.next_unit, 1);
      if (!push(cur < n_all ? cur : -1)) ok = false;
      while (ok && cur < n_all) {
        const int nxt = atomicAdd(a.next_unit, 1);  // hand out the next unit ahead
        const int i = cur;
        cur = nxt;
        const XUnit X = unit_at(a, i, n_gu);
        const Unit& U = X.u;
        const bool shared = U.g == kE;
        const int N = round_up(U.nrows, kRowAlign);
        if (!push(nxt < n_all ? nxt : -1)) { ok = false; break; }
        if constexpr (Q4) {
          // the unit's group scales and biases (one contiguous block per array: consecutive
          // rows) into L2 with its first codes, so that the dequantizing warps' loads hit L2
          if (!X.down) {
            const int G = a.d / kBK;
            const size_t r0 = (shared ? 0 : (size_t)U.g * a.f) + U.mt * kMTile;
            for (int m = 0; m < 2; ++m) {
              const int mat = (shared ? 3 : 0) + m;
              prefetch_l2_bulk(a.q4.s[mat] + r0 * G, kMTile * G * 2);
              prefetch_l2_bulk(a.q4.b[mat] + r0 * G, kMTile * G * 2);
            }
          } else {
            const int G = (shared ? a.fs : a.f) / kBK, mat = shared ? 5 : 2;
            const size_t r0 = (shared ? 0 : (size_t)U.g * a.d) + U.mt * 2 * kMTile;
            const int rows = (U.mt * 2 + 1) * kMTile < a.d ? 2 * kMTile : kMTile;
            prefetch_l2_bulk(a.q4.s[mat] + r0 * G, rows * G * 2);
            prefetch_l2_bulk(a.q4.b[mat] + r0 * G, rows * G * 2);
          }
        }
        if (!X.down) {
          const CUtensorMap* mg = shared ? &tm_wsg : &tm_wg;
          const CUtensorMap* mu = shared ? &tm_wsu : &tm_wu;
          const int arow = (shared ? 0 : U.g * a.f) + U.mt * kMTile;
          const uint64_t pw = shared ? keep_h : stream_w;
          for (int kb = 0; kb < a.d / kBK; ++kb) {
            if (!mbar_wait(&empty[stage], ph ^ 1, a.err)) { ok = false; break; }
            uint8_t* st = smem + stage * kXStage;
            if constexpr (Q4) {
              // codes of both tiles (x counts bytes: 32 per 64-input step); the token rows
              // arrive by cp.async, so full[] only gets this lane's plain arrival
              mbar_arrive_expect_tx(&cfull[stage], 2 * kQTile);
              tma_load_2d(st, mg, &cfull[stage], kb * (kBK / 2), arow, pw);
              tma_load_2d(st + kQTile, mu, &cfull[stage], kb * (kBK / 2), arow, pw);
              mbar_arrive(&full[stage]);
            } else {
              mbar_arrive_expect_tx(&full[stage], 2 * kTileA);
              tma_load_2d(st, mg, &full[stage], kb * kBK, arow, pw);
              tma_load_2d(st + kTileA, mu, &full[stage], kb * kBK, arow, pw);
            }
            if (++stage == kXStages) { stage = 0; ph ^= 1; }
          }
        } else {
          // the chunk's h rows are complete once all its gate/up tiles have published
          const int need = (shared ? a.fs : a.f) / kMTile;
          const uint64_t t0 = global_timer_ns();
          while (true) {
            int v;
            asm volatile("ld.acquire.gpu.global.b32 %0, [%1];"
                         : "=r"(v)
                         : "l"(a.chunk_done + U.cid)
                         : "memory");
            if (v >= need) break;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
              atomicExch(a.err, kDevErrTimeout);
              ok = false;
              break;
            }
          }
          if (!ok) break;
          asm volatile("fence.proxy.async.global;" ::: "memory");  // h read by TMA next
          // two 128-row tiles of the down weights (outputs mt*256 .. +255) share the h rows
          const int K = shared ? a.fs : a.f;
          const CUtensorMap* mw = shared ? &tm_wsd : &tm_wd;
          const int arow = (shared ? 0 : U.g * a.d) + U.mt * 2 * kMTile;
          const bool two = (U.mt * 2 + 1) * kMTile < a.d;
          // h rows in boxes of kHBoxRows (<= 3 boxes: N <= 192); the rows of the last box past
          // N land in B rows the MMA does not read (past the end of h the box is zero-filled)
          const int nbox = (N + kHBoxRows - 1) / kHBoxRows;
          const uint32_t hbytes = (uint32_t)nbox * kHBoxRows * kBK * 2;
          const uint32_t bytes = (Q4 ? 0 : (two ? 2 : 1) * kTileA) + hbytes;
          for (int kb = 0; kb < K / kBK; ++kb) {
            if (!mbar_wait(&empty[stage], ph ^ 1, a.err)) { ok = false; break; }
            uint8_t* st = smem + stage * kXStage;
            const uint64_t pw = shared ? keep_h : stream_w;
            if constexpr (Q4) {
              mbar_arrive_expect_tx(&cfull[stage], (two ? 2 : 1) * kQTile);
              tma_load_2d(st, mw, &cfull[stage], kb * (kBK / 2), arow, pw);
              if (two)
                tma_load_2d(st + kQTile, mw, &cfull[stage], kb * (kBK / 2), arow + kMTile, pw);
            }
            mbar_arrive_expect_tx(&full[stage], bytes);
            if constexpr (!Q4) {
              tma_load_2d(st, mw, &full[stage], kb * kBK, arow, pw);
              if (two) tma_load_2d(st + kTileA, mw, &full[stage], kb * kBK, arow + kMTile, pw);
            }
            for (int r = 0; r < nbox; ++r)
              tma_load_2d(st + C::kBOff + r * (kHBoxRows * kBK * 2), &tm_h, &full[stage],
                          kb * kBK, U.p0 + kHBoxRows * r, keep_h);
            if (++stage == kXStages) { stage = 0; ph ^= 1; }
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t ph = 0, tph[2] = {0, 0};
      int ab = 0;  // 4-bit: dequantized A buffer of the next stage
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int i = next_unit_1(k, ok);
        if (i < 0) break;
        const XUnit X = unit_at(a, i, n_gu);
        const Unit& U = X.u;
        const int N = round_up(U.nrows, kRowAlign);
        const uint32_t idesc = idesc_bf16(128, N);
        // both TMEM halves: gate (or down rows +0..127) in [0, N), up (or down rows
        // +128..255) in [256, 256 + N)
        const bool two = !X.down || (U.mt * 2 + 1) * kMTile < a.d;
        const int KB = X.down ? (U.g == kE ? a.fs : a.f) / kBK : a.d / kBK;
        if (!mbar_wait(&tempty[0], tph[0] ^ 1, a.err) ||
            !mbar_wait(&tempty[1], tph[1] ^ 1, a.err))
          break;
        tc_fence_after();
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&full[stage], ph, a.err)) { ok = false; break; }
          fence_proxy_async_smem();  // token rows of gate/up units come from cp.async
          tc_fence_after();
          const uint32_t s0 = smem_u32(smem + stage * kXStage);
          const uint32_t s1 = s0 + kTileA, sb = s0 + C::kBOff;
          if constexpr (Q4) {
            // A from tensor memory: 16 inputs = 8 columns per MMA, tile 1 at +32 columns
            const uint32_t a0 = tmem + abuf_col(ab);
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk) {
              const uint64_t bd = sdesc_k128(sb + kk * 32);
              const uint32_t acc = (kb | kk) != 0;
              mma_bf16_ts(tmem, a0 + kk * 8, bd, idesc, acc);
              if (two) mma_bf16_ts(tmem + 256, a0 + 32 + kk * 8, bd, idesc, acc);
            }
            mma_commit(&aempty[ab]);
            ab ^= 1;
          } else {
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk) {
              const uint64_t bd = sdesc_k128(sb + kk * 32);
              const uint32_t acc = (kb | kk) != 0;
              mma_bf16(tmem, sdesc_k128(s0 + kk * 32), bd, idesc, acc);
              if (two) mma_bf16(tmem + 256, sdesc_k128(s1 + kk * 32), bd, idesc, acc);
            }
          }
          mma_commit(&empty[stage]);
          if (++stage == kXStages) { stage = 0; ph ^= 1; }
        }
        if (!ok) break;
        mma_commit(&tfull[0]);
        mma_commit(&tfull[1]);
        tph[0] ^= 1;
        tph[1] ^= 1;
      }
    }
  } else if (warp < 4) {
    // ---- token rows of gate/up units: thread (crow, chunk) copies 16-byte chunk `chunk` of
    // rows crow + 8i; for down units the thread only arrives, keeping the ring's phases
    const int bt = threadIdx.x - 64;
    const int crow = bt >> 3, chunk = bt & 7;
    const uint32_t swz = (uint32_t)((chunk ^ crow) << 4);  // (r & 7) == crow for every row
    const uint64_t keep_x = policy_evict_last();            // x rows are gathered many times
    int stage = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int i = next_unit(k, ok);
      if (i < 0) break;
      const XUnit X = unit_at(a, i, n_gu);
      const Unit& U = X.u;
      const int N = round_up(U.nrows, kRowAlign);
      const int nr = N / 8;  // rows per thread, <= 32
      const int KB = X.down ? (U.g == kE ? a.fs : a.f) / kBK : a.d / kBK;
      const __nv_bfloat16* src[kChunkRows / 8];
      if (!X.down) {
#pragma unroll
        for (int r = 0; r < kChunkRows / 8; ++r)
          src[r] = a.x + (size_t)(r < nr ? __ldg(a.grow + U.p0 + crow + 8 * r) : 0) * a.d +
                   chunk * 8;
      }
      for (int kb = 0; kb < KB; ++kb) {
        const bool w = mbar_wait(&empty[stage], ph ^ 1, a.err);
        if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
        if (!X.down) {
          const uint32_t sb =
              smem_u32(smem + stage * kXStage + C::kBOff) + crow * 128 + swz;
#pragma unroll
          for (int r = 0; r < kChunkRows / 8; ++r)
            if (r < nr) cp_async_16(sb + r * 1024, src[r] + kb * kBK, keep_x);
          cp_async_arrive_noinc(&full[stage]);
        } else {
          mbar_arrive(&full[stage]);
        }
        if (++stage == kXStages) { stage = 0; ph ^= 1; }
      }
    }
  } else if (warp < 12) {
    // ---- epilogue: thread = one weight row of the tile; the two warps of a lane quadrant
    // take alternate 16-column chunks
    const int q = warp & 3, half = (warp - 4) >> 2;
    const int m = q * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const uint64_t pol_keep = policy_evict_last();  // ys: read back soon by the combine
    uint32_t tph[2] = {0, 0};
    bool ok = true;
    // the unit's accumulators are released as soon as this warp's last TMEM read of them has
    // completed, so that the next unit's MMAs overlap the last chunk's arithmetic and stores
    auto release = [&]() {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&tempty[0]);
        mbar_arrive(&tempty[1]);
      }
    };
    for (int k = 0; ok; ++k) {
      const int i = next_unit(k, ok);
      if (i < 0) break;
      const XUnit X = unit_at(a, i, n_gu);
      const Unit& U = X.u;
      const int N = round_up(U.nrows, kRowAlign);
      const bool w0 = mbar_wait(&tfull[0], tph[0], a.err);
      const bool w1 = mbar_wait(&tfull[1], tph[1], a.err);
      if (!__all_sync(0xffffffffu, w0 && w1)) break;
      tc_fence_after();
      if (half * 16 >= N) release();  // no columns for this warp in this unit
      if (!X.down) {
        __nv_bfloat16* hp = a.h + (size_t)U.p0 * a.hdim + U.mt * kMTile + m;
        for (int j0 = half * 16; j0 < N; j0 += 32) {
          uint32_t g[16], v[16];
          tmem_ld16(tmem + lane_off + (uint32_t)j0, g);
          tmem_ld16(tmem + lane_off + 256u + (uint32_t)j0, v);
          tmem_wait_ld();
          if (j0 + 32 >= N) release();
#pragma unroll
          for (int r = 0; r < 16; ++r)
            hp[(size_t)(j0 + r) * a.hdim] =
                __float2bfloat16_rn(silu_mul(__uint_as_float(g[r]), __uint_as_float(v[r])));
        }
        tph[0] ^= 1;
        tph[1] ^= 1;
        // publish: all epilogue warps' h stores of this unit, then the chunk counter
        named_sync(2, kXEpiWarps * 32);
        if (threadIdx.x == 128) {
          __threadfence();
          atomicAdd(a.chunk_done + U.cid, 1);
        }
      } else {
        const bool two = (U.mt * 2 + 1) * kMTile < a.d;
        __nv_bfloat16* yp = a.ys + (size_t)U.p0 * a.d + U.mt * 2 * kMTile + m;
        for (int j0 = half * 16; j0 < N; j0 += 32) {
          uint32_t r0[16], r1[16];
          tmem_ld16(tmem + lane_off + (uint32_t)j0, r0);
          if (two) tmem_ld16(tmem + lane_off + 256u + (uint32_t)j0, r1);
          tmem_wait_ld();
          if (j0 + 32 >= N) release();
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            st_b16_hint(yp + (size_t)(j0 + c) * a.d, __float2bfloat16_rn(__uint_as_float(r0[c])),
                        pol_keep);
            if (two)
              st_b16_hint(yp + (size_t)(j0 + c) * a.d + kMTile,
                          __float2bfloat16_rn(__uint_as_float(r1[c])), pol_keep);
          }
        }
        tph[0] ^= 1;
        tph[1] ^= 1;
      }
    }
  } else if constexpr (Q4) {
    // ---- dequantization: two groups of four warps take alternate pipeline steps (group g
    // the steps that fill A buffer g; with an even number of ring stages each group always
    // uses the same ring slots), so a warp has two step periods for its step.  Thread = row r
    // of both tiles (gate and up, or the two down tiles) in the lane quadrant its warp may
    // address.  Per step and tile: the row's 64 codes (32 bytes) from shared memory, one scale
    // and one bias, 32 columns of bf16 pairs into the A buffer in tensor memory.
    static_assert(kXStages % 2 == 0, "each dequantization group keeps its own ring slots");
    const int q = warp & 3, grp = (warp - 12) >> 2;
    const int r = q * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const uint32_t acol = abuf_col(grp);
    int stage = grp, n = 0;  // this group's next ring slot; steps of the units before (both groups)
    uint32_t ph = 0, aph = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int i = next_unit(k, ok);
      if (i < 0) break;
      const XUnit X = unit_at(a, i, n_gu);
      const Unit& U = X.u;
      const bool shared = U.g == kE;
      int K, mat0, mat1;
      size_t row0, row1;
      if (!X.down) {
        K = a.d;
        mat0 = shared ? 3 : 0;
        mat1 = mat0 + 1;
        row0 = row1 = (shared ? 0 : (size_t)U.g * a.f) + U.mt * kMTile + r;
      } else {
        K = shared ? a.fs : a.f;
        mat0 = mat1 = shared ? 5 : 2;
        row0 = (shared ? 0 : (size_t)U.g * a.d) + U.mt * 2 * kMTile + r;
        row1 = row0 + kMTile;
      }
      // a down unit whose outputs end inside its first tile has no second tile
      const bool two = !X.down || (U.mt * 2 + 1) * kMTile < a.d;
      const int G = K / kBK;
      const unsigned short* sp0 = reinterpret_cast<const unsigned short*>(a.q4.s[mat0]) + row0 * G;
      const unsigned short* bp0 = reinterpret_cast<const unsigned short*>(a.q4.b[mat0]) + row0 * G;
      const unsigned short* sp1 = reinterpret_cast<const unsigned short*>(a.q4.s[mat1]) + row1 * G;
      const unsigned short* bp1 = reinterpret_cast<const unsigned short*>(a.q4.b[mat1]) + row1 * G;
      // this group's steps of the unit: kb = kb0, kb0 + 2, ...; each step's scales and biases
      // are loaded one step of the group ahead
      int kb = (grp ^ n) & 1;
      n += G;
      uint32_t s0 = 0, b0 = 0, s1 = 0, b1 = 0;
      if (kb < G) {
        s0 = __ldg(sp0 + kb);
        b0 = __ldg(bp0 + kb);
        if (two) {
          s1 = __ldg(sp1 + kb);
          b1 = __ldg(bp1 + kb);
        }
      }
      for (; kb < G; kb += 2) {
        uint32_t ns0 = 0, nb0 = 0, ns1 = 0, nb1 = 0;
        if (kb + 2 < G) {
          ns0 = __ldg(sp0 + kb + 2);
          nb0 = __ldg(bp0 + kb + 2);
          if (two) {
            ns1 = __ldg(sp1 + kb + 2);
            nb1 = __ldg(bp1 + kb + 2);
          }
        }
        bool w = mbar_wait(&cfull[stage], ph, a.err);
        if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
        const uint8_t* cbase = smem + stage * kXStage + r * 32;
        uint32_t v[32];
        dequant_q4_row(reinterpret_cast<const uint4*>(cbase), s0, b0, v);
        w = mbar_wait(&aempty[grp], aph ^ 1, a.err);  // the MMA has read this A buffer
        if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
        tc_fence_after();
        tmem_st32(tmem + lane_off + acol, v);
        if (two) {
          dequant_q4_row(reinterpret_cast<const uint4*>(cbase + kQTile), s1, b1, v);
          tmem_st32(tmem + lane_off + acol + 32u, v);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[stage]);
        stage += 2;
        if (stage >= kXStages) { stage -= kXStages; ph ^= 1; }
        aph ^= 1;
        s0 = ns0;
        b0 = nb0;
        s1 = ns1;
        b1 = nb1;
      }
    }
  }
  pdl_trigger();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------- combine

constexpr int kCbCols = 2048;               // output columns per combine unit (256 threads x 8)
constexpr int kCbStages = 6;
constexpr int kCbStage = 9 * kCbCols * 2;   // the nine ys rows of one unit (36 KB)
constexpr int kCbThreads = 288;             // warps 0-7 combine, warp 8 copies
constexpr int kCbSmem = kCbStages * kCbStage + 256;

// y[t] = sum over j = 0..7 (ascending expert id) of w_j * ys[prow[t][j]], then
// + ys[prow[t][8]] (the shared expert), in fp32, rounded once to bf16.
// Persistent blocks (one per SM) walk the units (token t, slice of up to 2048 columns) in a
// static round robin.  Warp 8 stages the unit's nine ys rows in shared memory with bulk async
// copies (one row per lane, six units in flight, so that enough bytes are in flight to cover
// the HBM latency), and the eight combine warps take 8 consecutive outputs per thread.
__global__ void __launch_bounds__(kCbThreads, 1)
    combine_kernel(int T, int d, const float* topk_w, const int32_t* prow,
                   const __nv_bfloat16* ys, __nv_bfloat16* y, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((128 - (smem_u32(smem_raw) & 127)) & 127);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kCbStages * kCbStage);
  uint64_t* empty = full + kCbStages;
  __shared__ int s_fail;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kCbStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 8);
    }
    s_fail = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();  // prow, topk_w and ys come from earlier kernels on the stream
  const int nslice = (d + kCbCols - 1) / kCbCols;
  const int n_units = T * nslice;
  const int G = (int)gridDim.x;
  int k = 0;
  if (warp == 8) {
    const uint64_t pol = policy_evict_first();  // last use of ys
    // the row indices of three units are loaded at once (lane 9 i + j: row j of unit i), one
    // batch ahead of the copies, so the copy issue never waits on them
    const int bi = lane / 9, bj = lane % 9;
    auto rows_of = [&](int ub) {
      const int u = ub + bi * G;
      return lane < 27 && u < n_units ? __ldg(prow + (size_t)(u / nslice) * 9 + bj) : 0;
    };
    int rcur = rows_of(blockIdx.x);
    bool ok = true;
    for (int ub = blockIdx.x; ok && ub < n_units; ub += 3 * G) {
      const int rnext = rows_of(ub + 3 * G);
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        const int u = ub + i * G;
        if (u >= n_units) break;
        const int r = __shfl_sync(0xffffffffu, rcur, i * 9 + (lane < 9 ? lane : 0));
        const int st = k % kCbStages;
        const int c0 = (u % nslice) * kCbCols;
        const int cols = min(kCbCols, d - c0);
        ok = __all_sync(0xffffffffu, mbar_wait(&empty[st], ((k / kCbStages) & 1) ^ 1, err));
        if (!ok) { s_fail = 1; break; }
        if (lane == 0) mbar_arrive_expect_tx(&full[st], 9u * cols * 2);
        __syncwarp();
        if (lane < 9)
          bulk_load(smem + st * kCbStage + lane * (kCbCols * 2), ys + (size_t)r * d + c0,
                    (uint32_t)cols * 2, &full[st], pol);
        ++k;
      }
      rcur = rnext;
    }
  } else {
    const int c = threadIdx.x * 8;
    for (int u = blockIdx.x; u < n_units; u += G, ++k) {
      const int st = k % kCbStages;
      const int t = u / nslice, c0 = (u % nslice) * kCbCols;
      const int cols = min(kCbCols, d - c0);
      const float4 wa = __ldg(reinterpret_cast<const float4*>(topk_w + (size_t)t * kTopK));
      const float4 wb = __ldg(reinterpret_cast<const float4*>(topk_w + (size_t)t * kTopK) + 1);
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&full[st], (k / kCbStages) & 1, err));
      if (!ok) { s_fail = 1; break; }
      if (c < cols) {
        const float w[9] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w, 1.0f};
        const uint8_t* row = smem + st * kCbStage + c * 2;
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
        for (int j = 0; j < 9; ++j) {
          const uint4 v = *reinterpret_cast<const uint4*>(row + j * (kCbCols * 2));
          const uint32_t p[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[2 * i] += w[j] * bf16_lo(p[i]);
            acc[2 * i + 1] += w[j] * bf16_hi(p[i]);
          }
        }
        uint4 o;
        uint32_t* po = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
          po[i] = *reinterpret_cast<uint32_t*>(&b2);
        }
        *reinterpret_cast<uint4*>(y + (size_t)t * d + c0 + c) = o;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
  }
  pdl_trigger();
  __syncthreads();
  // after a timed-out wait, let the copies already issued land (bounded) before exiting
  if (s_fail && warp == 8 && lane == 0)
    for (int kk = k > kCbStages ? k - kCbStages : 0; kk < k; ++kk)
      mbar_wait(&full[kk % kCbStages], (kk / kCbStages) & 1, err);
}

}  // namespace

cudaError_t prepare_expert_kernels() {
  cudaError_t e = cudaFuncSetAttribute(experts_kernel<false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       XCfg<false>::kSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(experts_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           XCfg<true>::kSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kCbSmem);
}

cudaError_t launch_experts(const __nv_bfloat16* x, const CUtensorMap& tm_wg,
                           const CUtensorMap& tm_wu, const CUtensorMap& tm_wsg,
                           const CUtensorMap& tm_wsu, const CUtensorMap& tm_h,
                           const CUtensorMap& tm_wd, const CUtensorMap& tm_wsd, const Dims& D,
                           const RouteWs& ws, __nv_bfloat16* h, __nv_bfloat16* ys, int grid,
                           cudaStream_t s, const Q4Weights* q4) {
  XArgs a{ws.units_gu, ws.units_dn, ws.n_units, ws.next_unit, ws.chunk_done, ws.grow, x, h, ys,
          D.d, D.f, D.fs, D.hdim, ws.err, XQ4{}};
  if (!q4)
    return launch_pdl(experts_kernel<false>, dim3(grid), dim3(XCfg<false>::kThreads),
                      XCfg<false>::kSmem, s, tm_wg, tm_wu, tm_wsg, tm_wsu, tm_h, tm_wd, tm_wsd, a);
  const Q4Matrix* m[6] = {&q4->gate, &q4->up, &q4->down, &q4->s_gate, &q4->s_up, &q4->s_down};
  for (int i = 0; i < 6; ++i) {
    a.q4.s[i] = m[i]->scales;
    a.q4.b[i] = m[i]->biases;
  }
  return launch_pdl(experts_kernel<true>, dim3(grid), dim3(XCfg<true>::kThreads),
                    XCfg<true>::kSmem, s, tm_wg, tm_wu, tm_wsg, tm_wsu, tm_h, tm_wd, tm_wsd, a);
}

cudaError_t launch_combine(int T, const Dims& D, const float* topk_w, const RouteWs& ws,
                           const __nv_bfloat16* ys, __nv_bfloat16* y, int grid, cudaStream_t s) {
  const int units = T * ((D.d + kCbCols - 1) / kCbCols);
  return launch_pdl(combine_kernel, dim3(units < grid ? units : grid), dim3(kCbThreads), kCbSmem,
                    s, T, D.d, topk_w, (const int32_t*)ws.prow, ys, y, ws.err);
}

}  // namespace moe
