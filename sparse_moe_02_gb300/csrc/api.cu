// The C ABI of libmoe (declared and documented in include/moe.h): argument checks, the
// device workspace, TMA tensor maps, and the order of the kernel launches of one layer.
// Nothing here synchronises with the host inside moe_route / moe_forward.
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "layer.cuh"
#include "moe.h"

using moe::Dims;
using moe::kE;
using moe::kTopK;

namespace {

thread_local int g_last_cuda_error = 0;

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  g_last_cuda_error = (int)e;
  return MOE_ERR_CUDA;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D bf16 tensor [rows][inner] (row pitch inner*2 bytes), box [box_rows][box_inner],
// 128-byte swizzle (the layout the tcgen05 descriptors expect).
bool encode_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
               uint32_t box_inner, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D byte tensor [rows][inner] of 4-bit codes (row pitch inner bytes), box [128 rows][32
// bytes] = one 64-input step of a 128-row tile, no swizzle.
bool encode_codes(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner};
  cuuint32_t box[2] = {moe::kBK / 2, moe::kMTile};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The device address of page-locked host memory the device can address, if p is such memory
// and 16-byte aligned there; else NULL (pageable memory, or a pointer CUDA does not know).
void* device_view(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (at.type != cudaMemoryTypeHost || !at.devicePointer || !aligned16(at.devicePointer))
    return nullptr;
  return at.devicePointer;
}
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

struct moe_handle_s {
  moe_config cfg;
  moe_weights w;       // bf16 handle: the weights; 4-bit handle: only w_router, router_bias
  bool q4 = false;     // 4-bit experts
  moe::Q4Weights wq{};
  Dims D;
  int device = 0, sms = 0;
  int P_max = 0, max_units_gu = 0, max_units_dn = 0, max_chunks = 0;
  int Tc = 0, P_chunk = 0;  // tokens per forward chunk; rows of h and ys for one chunk
  void* ws = nullptr;
  size_t ws_bytes = 0;
  moe::RouteWs rws{};
  moe::DecodeWs dws{};
  __nv_bfloat16* h = nullptr;
  __nv_bfloat16* ys = nullptr;
  __nv_bfloat16* x_stage = nullptr;
  __nv_bfloat16* y_stage = nullptr;
  CUtensorMap tm_wr, tm_wg, tm_wu, tm_wsg, tm_wsu, tm_wd, tm_wsd, tm_h;
  // per-kernel timing (moe_profile_begin / moe_profile_end)
  static constexpr int kMaxKernels = 6;
  std::vector<cudaEvent_t> prof_ev;  // [n_calls][kMaxKernels + 1]
  int prof_calls = 0, prof_done = 0, prof_nk = 0;
  int expire_calls = 0;  // moe_test_expire_waits: streamed decode launches left to expire
};

namespace {

int check_config(const moe_config* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->d <= 0 || c->ffn_dim <= 0 || c->shared_ffn_dim <= 0 || c->max_tokens <= 0 ||
      c->n_experts <= 0 || c->top_k <= 0)
    return MOE_ERR_INVALID_ARG;
  if (c->schedule < MOE_SCHEDULE_AUTO || c->schedule > MOE_SCHEDULE_GEMV)
    return MOE_ERR_INVALID_ARG;
  if (c->n_experts != kE || c->top_k != kTopK) return MOE_ERR_UNSUPPORTED;
  if (c->d % 128 || c->d > 8192) return MOE_ERR_UNSUPPORTED;
  if (c->ffn_dim % 128 || c->ffn_dim > 2048) return MOE_ERR_UNSUPPORTED;
  if (c->shared_ffn_dim % 128 || c->shared_ffn_dim > 2048) return MOE_ERR_UNSUPPORTED;
  if (c->max_tokens > (1 << 20)) return MOE_ERR_UNSUPPORTED;
  if (c->chunk_tokens < 0) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

int check_weights(const moe_weights* w) {
  if (!w) return MOE_ERR_INVALID_ARG;
  const void* req[] = {w->w_router, w->w_gate, w->w_up, w->w_down, w->ws_gate, w->ws_up,
                       w->ws_down};
  for (const void* p : req) {
    if (!p) return MOE_ERR_INVALID_ARG;
    if (!aligned16(p)) return MOE_ERR_ALIGNMENT;
  }
  if (w->router_bias && !aligned4(w->router_bias)) return MOE_ERR_ALIGNMENT;
  return MOE_OK;
}

int check_q4(const moe_weights_q4* w) {
  if (!w || !w->w_router) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w->w_router)) return MOE_ERR_ALIGNMENT;
  if (w->router_bias && !aligned4(w->router_bias)) return MOE_ERR_ALIGNMENT;
  const moe_q4_matrix* ms[] = {&w->w_gate, &w->w_up, &w->w_down, &w->ws_gate, &w->ws_up,
                               &w->ws_down};
  for (const moe_q4_matrix* m : ms) {
    if (!m->codes || !m->scales || !m->biases) return MOE_ERR_INVALID_ARG;
    if (!aligned16(m->codes) || !aligned16(m->scales) || !aligned16(m->biases))
      return MOE_ERR_ALIGNMENT;
  }
  return MOE_OK;
}

moe::Q4Matrix q4_matrix(const moe_q4_matrix& m) {
  return moe::Q4Matrix{static_cast<const uint8_t*>(m.codes),
                       static_cast<const __nv_bfloat16*>(m.scales),
                       static_cast<const __nv_bfloat16*>(m.biases)};
}

// Bump allocator over the single workspace allocation (256-byte aligned pieces).
struct Carve {
  char* base;
  size_t off = 0;
  template <typename T>
  T* take(size_t n) {
    off = (off + 255) & ~size_t(255);
    T* p = reinterpret_cast<T*>(base ? base + off : nullptr);
    off += n * sizeof(T);
    return p;
  }
};

void layout(moe_handle_s* h, char* base, size_t* total) {
  const int Tm = h->cfg.max_tokens;
  const int nblk = (Tm + moe::kBlockTokens - 1) / moe::kBlockTokens;
  const size_t S = (size_t)Tm * kTopK;
  Carve c{base};
  h->rws.topk_idx = c.take<int32_t>(S);
  h->rws.topk_w = c.take<float>(S);
  h->rws.hist = c.take<int32_t>((size_t)nblk * kE);
  h->rws.blkpre = c.take<int32_t>((size_t)nblk * kE);
  h->rws.offsets = c.take<int32_t>(kE + 1);
  h->rws.poff = c.take<int32_t>(kE + 2);
  h->rws.perm = c.take<int32_t>(S);
  h->rws.prow = c.take<int32_t>((size_t)Tm * 9);
  h->rws.grow = c.take<int32_t>((size_t)h->P_max);
  h->rws.units_gu = c.take<moe::Unit>((size_t)h->max_units_gu);
  h->rws.units_dn = c.take<moe::Unit>((size_t)h->max_units_dn);
  h->rws.n_units = c.take<int32_t>(2);
  h->rws.next_unit = c.take<int32_t>(1);
  h->rws.chunk_done = c.take<int32_t>((size_t)h->max_chunks);
  h->rws.err = c.take<int>(1);
  h->dws.logits = c.take<float>((size_t)moe::kGemvMaxTokens * kE);
  h->dws.counter = c.take<int>(1);
  h->dws.gu_next = c.take<int>(1);
  h->dws.hdec = c.take<float>((size_t)moe::kGemvMaxTokens * 9 * h->D.hdim);
  // the large per-slot buffers hold one forward chunk (Tc tokens, P_chunk padded rows)
  h->h = c.take<__nv_bfloat16>((size_t)h->P_chunk * h->D.hdim);
  h->ys = c.take<__nv_bfloat16>((size_t)h->P_chunk * h->D.d);
  h->x_stage = c.take<__nv_bfloat16>((size_t)h->Tc * h->D.d);
  h->y_stage = c.take<__nv_bfloat16>((size_t)h->Tc * h->D.d);
  *total = c.off + 256;
}

moe::DecodeWeights decode_weights(const moe_handle_s* h) {
  moe::DecodeWeights W;
  W.w_r = static_cast<const __nv_bfloat16*>(h->w.w_router);
  W.w_gate = static_cast<const __nv_bfloat16*>(h->w.w_gate);
  W.w_up = static_cast<const __nv_bfloat16*>(h->w.w_up);
  W.w_down = static_cast<const __nv_bfloat16*>(h->w.w_down);
  W.ws_gate = static_cast<const __nv_bfloat16*>(h->w.ws_gate);
  W.ws_up = static_cast<const __nv_bfloat16*>(h->w.ws_up);
  W.ws_down = static_cast<const __nv_bfloat16*>(h->w.ws_down);
  W.bias = h->w.router_bias;
  return W;
}

int check_call(moe_handle h, const void* x, int T) {
  if (!h) return MOE_ERR_INVALID_ARG;
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (T > h->cfg.max_tokens) return MOE_ERR_UNSUPPORTED;
  if (T > 0 && !x) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x)) return MOE_ERR_ALIGNMENT;
  // the small-batch matrix-vector path reads bf16 experts only
  if (h->cfg.schedule == MOE_SCHEDULE_GEMV && T > 1 &&
      (h->q4 || !moe::decode_batch_fits(h->D, T)))
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// Records the profiling event before kernel i (or after the last kernel, i = nk) of the
// current call when profiling is on.
int prof_mark(moe_handle h, cudaStream_t s, int i) {
  if (h->prof_done >= h->prof_calls) return MOE_OK;
  return cuda_status(cudaEventRecord(
      h->prof_ev[(size_t)h->prof_done * (moe_handle_s::kMaxKernels + 1) + i], s));
}

int prof_finish_call(moe_handle h, cudaStream_t s, int nk) {
  if (h->prof_done >= h->prof_calls) return MOE_OK;
  int st = prof_mark(h, s, nk);
  h->prof_nk = nk;
  ++h->prof_done;
  return st;
}

bool use_gemv(const moe_handle_s* h, int T) {
  return T == 1 && h->cfg.schedule != MOE_SCHEDULE_GEMM;
}

// Two tokens under AUTO with bf16 experts: one single-token pass per token, measured faster on
// GB300 than the grouped GEMM over both tokens or one pass over the union of their experts.
// Each token's routing is bit-identical to moe_route's (the batch router accumulates each
// token's logits in the single-token router's order and selects with the same routine).
bool per_token(const moe_handle_s* h, int T) {
  return T == 2 && h->cfg.schedule == MOE_SCHEDULE_AUTO && !h->q4;
}

// 2..8 tokens whose shapes fit, on request (schedule GEMV): the matrix-vector path over the
// union of their experts.  AUTO keeps T = 3..8 on the tensor-core path and runs T = 2 as one
// single-token pass per token, both measured faster on GB300 (bench.py's small-batch lines
// time all three).
bool use_batch(const moe_handle_s* h, int T) {
  return h->cfg.schedule == MOE_SCHEDULE_GEMV && moe::decode_batch_fits(h->D, T);
}

// Calls whose whole token count is this small take the matrix-vector router (a warp per
// router row over every SM, selection in the last block) instead of the tensor-core router,
// whose single 128-token block would stream the whole router matrix through four SMs.
// Decided on the call's T, not a chunk's, so that chunked calls route like unchunked ones.
bool small_router(const moe_handle_s* h, int T) {
  return T <= moe::kGemvMaxTokens && moe::decode_batch_fits(h->D, T);
}

// The routing chain of the tensor-core schedule (small: see small_router).
int run_route_gemm(moe_handle h, const void* x, int T, int32_t* topk_idx, float* topk_w,
                   int32_t* offsets, int32_t* perm, cudaStream_t s, bool prof, bool small) {
  moe::RouteWs w = h->rws;
  if (offsets) w.offsets = offsets;
  int st;
  if (prof && (st = prof_mark(h, s, 0))) return st;
  if (small) {
    // routing and the plan in one launch (the plan's profiling slot stays empty)
    if ((st = cuda_status(moe::launch_decode_batch_router_shared(
             static_cast<const __nv_bfloat16*>(x), decode_weights(h), h->D, T, topk_idx, topk_w,
             nullptr, perm, h->dws, s, false, &w))))
      return st;
    if (prof && (st = prof_mark(h, s, 1))) return st;
    return MOE_OK;
  } else {
    CUtensorMap tm_x;  // the router loads x in tiles of 128 rows x 64
    if (!encode_2d(&tm_x, x, h->D.d, T, moe::kBK, moe::kBlockTokens)) return MOE_ERR_CUDA;
    if ((st = cuda_status(moe::launch_router_topk(tm_x, h->tm_wr, h->w.router_bias, T, h->D,
                                                  topk_idx, topk_w, w, s))))
      return st;
  }
  if (prof && (st = prof_mark(h, s, 1))) return st;
  return cuda_status(moe::launch_route_plan_scatter(T, h->D, topk_idx, perm, w, s));
}

// The tensor-core schedule over T <= Tc tokens: routing chain, grouped GEMMs, combine
// (profiling marks 0..4 when prof).
int forward_gemm(moe_handle h, const __nv_bfloat16* xd, int T, __nv_bfloat16* yd,
                 cudaStream_t s, bool prof, bool small) {
  int st;
  if ((st = run_route_gemm(h, xd, T, h->rws.topk_idx, h->rws.topk_w, nullptr, h->rws.perm, s,
                           prof, small)))
    return st;
#ifdef MOE_DEBUG
  // debug build: the routing's invariants, into the device error word
  if ((st = cuda_status(moe::launch_check_routing(h->rws.topk_idx, h->rws.offsets, h->rws.perm, T,
                                                  h->rws.err, s))))
    return st;
#endif
  if (prof && (st = prof_mark(h, s, 2))) return st;
  if ((st = cuda_status(moe::launch_experts(xd, h->tm_wg, h->tm_wu, h->tm_wsg, h->tm_wsu,
                                            h->tm_h, h->tm_wd, h->tm_wsd, h->D, h->rws, h->h,
                                            h->ys, h->sms, s, h->q4 ? &h->wq : nullptr))))
    return st;
  if (prof && (st = prof_mark(h, s, 3))) return st;
  return cuda_status(moe::launch_combine(T, h->D, h->rws.topk_w, h->rws, h->ys, yd, h->sms, s));
}

// moe_create and moe_create_q4: exactly one of w (bf16 experts) and wq (4-bit experts).
int create_handle(const moe_config* cfg, const moe_weights* w, const moe_weights_q4* wq,
                  moe_handle* out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  int st = check_config(cfg);
  if (st) return st;
  if ((st = w ? check_weights(w) : check_q4(wq))) return st;

  moe_handle_s* h = new (std::nothrow) moe_handle_s();
  if (!h) return MOE_ERR_NO_MEMORY;
  h->cfg = *cfg;
  if (w) {
    h->w = *w;
  } else {
    h->q4 = true;
    h->w = moe_weights{};
    h->w.w_router = wq->w_router;
    h->w.router_bias = wq->router_bias;
    h->wq = moe::Q4Weights{static_cast<const __nv_bfloat16*>(wq->w_router), wq->router_bias,
                           q4_matrix(wq->w_gate), q4_matrix(wq->w_up), q4_matrix(wq->w_down),
                           q4_matrix(wq->ws_gate), q4_matrix(wq->ws_up),
                           q4_matrix(wq->ws_down)};
  }
  h->D = Dims{cfg->d, cfg->ffn_dim, cfg->shared_ffn_dim,
              cfg->ffn_dim > cfg->shared_ffn_dim ? cfg->ffn_dim : cfg->shared_ffn_dim};
  auto fail = [&](int status) {
    if (h->ws) cudaFree(h->ws);
    delete h;
    return status;
  };
  cudaDeviceProp prop;
  if ((st = cuda_status(cudaGetDevice(&h->device)))) return fail(st);
  if ((st = cuda_status(cudaGetDeviceProperties(&prop, h->device)))) return fail(st);
  if (prop.major != 10 || prop.minor != 3) return fail(MOE_ERR_UNSUPPORTED);  // sm_103 only
  h->sms = prop.multiProcessorCount;

  const int Tm = cfg->max_tokens;
  const int S = Tm * kTopK;
  // every group padded to 16 rows: routed groups add at most 15 rows each
  h->P_max = moe::round_up(S + kE * (moe::kRowAlign - 1) + moe::round_up(Tm, moe::kRowAlign), 256);
  h->Tc = cfg->chunk_tokens > 0 && cfg->chunk_tokens < Tm ? cfg->chunk_tokens : Tm;
  h->P_chunk = moe::round_up(h->Tc * kTopK + kE * (moe::kRowAlign - 1) +
                                 moe::round_up(h->Tc, moe::kRowAlign),
                             256);
  const int chunks_routed = (S + moe::kChunkRows - 1) / moe::kChunkRows + kE;
  const int chunks_shared = (Tm + moe::kChunkRows - 1) / moe::kChunkRows;
  h->max_units_gu = chunks_routed * (cfg->ffn_dim / moe::kMTile) +
                    chunks_shared * (cfg->shared_ffn_dim / moe::kMTile);
  h->max_units_dn = (chunks_routed + chunks_shared) * (cfg->d / moe::kMTile);
  h->max_chunks = chunks_routed + chunks_shared;

  size_t total = 0;
  layout(h, nullptr, &total);
  if (cudaMalloc(&h->ws, total) != cudaSuccess) {
    cudaGetLastError();
    return fail(MOE_ERR_NO_MEMORY);
  }
  h->ws_bytes = total;
  layout(h, static_cast<char*>(h->ws), &total);
  // zero everything once: error word, decode counter, padding rows of h and grow
  if ((st = cuda_status(cudaMemset(h->ws, 0, total)))) return fail(st);

  const Dims& D = h->D;
  bool ok = encode_2d(&h->tm_wr, h->w.w_router, D.d, kE, moe::kBK, kE) &&
            encode_2d(&h->tm_h, h->h, D.hdim, h->P_chunk, moe::kBK, moe::kHBoxRows);
  // the tensor-core path's maps of the experts: 4-bit code bytes, or bf16 tiles
  if (h->q4) {
    const moe::Q4Weights& q = h->wq;
    ok = ok && encode_codes(&h->tm_wg, q.gate.codes, D.d / 2, (uint64_t)kE * D.f) &&
         encode_codes(&h->tm_wu, q.up.codes, D.d / 2, (uint64_t)kE * D.f) &&
         encode_codes(&h->tm_wsg, q.s_gate.codes, D.d / 2, D.fs) &&
         encode_codes(&h->tm_wsu, q.s_up.codes, D.d / 2, D.fs) &&
         encode_codes(&h->tm_wd, q.down.codes, D.f / 2, (uint64_t)kE * D.d) &&
         encode_codes(&h->tm_wsd, q.s_down.codes, D.fs / 2, D.d);
  }
  ok = ok && (h->q4 ||
             (encode_2d(&h->tm_wg, w->w_gate, D.d, (uint64_t)kE * D.f, moe::kBK, moe::kMTile) &&
            encode_2d(&h->tm_wu, w->w_up, D.d, (uint64_t)kE * D.f, moe::kBK, moe::kMTile) &&
            encode_2d(&h->tm_wsg, w->ws_gate, D.d, D.fs, moe::kBK, moe::kMTile) &&
            encode_2d(&h->tm_wsu, w->ws_up, D.d, D.fs, moe::kBK, moe::kMTile) &&
            encode_2d(&h->tm_wd, w->w_down, D.f, (uint64_t)kE * D.d, moe::kBK, moe::kMTile) &&
            encode_2d(&h->tm_wsd, w->ws_down, D.fs, D.d, moe::kBK, moe::kMTile)));
  if (!ok) return fail(MOE_ERR_CUDA);
  if ((st = cuda_status(moe::prepare_route_kernels()))) return fail(st);
  if ((st = cuda_status(moe::prepare_expert_kernels()))) return fail(st);
  if ((st = cuda_status(moe::prepare_decode_kernels(D.hdim)))) return fail(st);
  if ((st = cuda_status(moe::prepare_decode_batch_kernels()))) return fail(st);
  if ((st = cuda_status(moe::prepare_decode_stream_kernels()))) return fail(st);
  if ((st = cuda_status(moe::prepare_decode_q4_kernels()))) return fail(st);
  if ((st = cuda_status(cudaDeviceSynchronize()))) return fail(st);
  *out = h;
  return MOE_OK;
}

}  // namespace

extern "C" {

int moe_create(const moe_config* cfg, const moe_weights* w, moe_handle* out) {
  if (!w) {
    if (out) *out = nullptr;
    return MOE_ERR_INVALID_ARG;
  }
  return create_handle(cfg, w, nullptr, out);
}

int moe_create_q4(const moe_config* cfg, const moe_weights_q4* w, moe_handle* out) {
  if (!w) {
    if (out) *out = nullptr;
    return MOE_ERR_INVALID_ARG;
  }
  return create_handle(cfg, nullptr, w, out);
}

int moe_route(moe_handle h, const void* x, int T, int32_t* topk_idx, float* topk_w,
              int32_t* offsets, int32_t* perm, void* stream) {
  int st = check_call(h, x, T);
  if (st) return st;
  if (!aligned16(topk_idx) || !aligned16(topk_w) || !aligned4(offsets) || !aligned4(perm))
    return MOE_ERR_ALIGNMENT;
  if (T == 0) return MOE_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* idx = topk_idx ? topk_idx : h->rws.topk_idx;
  float* wt = topk_w ? topk_w : h->rws.topk_w;
  int32_t* pm = perm ? perm : h->rws.perm;
  int32_t* off = offsets ? offsets : h->rws.offsets;
  if (use_gemv(h, T))
    st = cuda_status(moe::launch_decode_router_shared(
        static_cast<const __nv_bfloat16*>(x), decode_weights(h), h->D, idx, wt, off, pm, h->dws,
        h->rws.err, s, false));
  else if (!h->q4 && use_batch(h, T))
    st = cuda_status(moe::launch_decode_batch_router_shared(
        static_cast<const __nv_bfloat16*>(x), decode_weights(h), h->D, T, idx, wt, off, pm,
        h->dws, s, false));
  else
    st = run_route_gemm(h, x, T, idx, wt, offsets, pm, s, false, small_router(h, T));
#ifdef MOE_DEBUG
  // debug build: the routing's invariants, into the device error word
  if (st == MOE_OK)
    st = cuda_status(moe::launch_check_routing(idx, off, pm, T, h->rws.err, s));
#endif
  return st;
}

int moe_forward(moe_handle h, const void* x, int T, void* y, void* stream) {
  int st = check_call(h, x, T);
  if (st) return st;
  if (T > 0 && !y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y)) return MOE_ERR_ALIGNMENT;
  if (T == 0) return MOE_OK;
  const size_t bytes = (size_t)T * h->D.d * 2;
  const char *xb = static_cast<const char*>(x), *yb = static_cast<const char*>(y);
  if (xb < yb + bytes && yb < xb + bytes) return MOE_ERR_INVALID_ARG;  // y overlaps x
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const __nv_bfloat16* xd = static_cast<const __nv_bfloat16*>(x);
  __nv_bfloat16* yd = static_cast<__nv_bfloat16*>(y);

  if (h->q4 && use_gemv(h, T)) {  // 4-bit experts, batch-1 decode
    if ((st = prof_mark(h, s, 0))) return st;
    // the router is bf16 on 4-bit handles too: the bf16 path's router launch, so that the
    // routing equals moe_route's bit for bit
    if ((st = cuda_status(moe::launch_decode_router_shared(xd, decode_weights(h), h->D, nullptr,
                                                           nullptr, nullptr, nullptr, h->dws,
                                                           h->rws.err, s, false))))
      return st;
    if ((st = prof_mark(h, s, 1))) return st;
    if (moe::decode_stream_fits(h->D, h->sms, true)) {
      // selection, gate/up and down with the combine in one launch (profiling slot 2 empty)
      if ((st = cuda_status(moe::launch_decode_stream(xd, decode_weights(h), h->D,
                                                      h->rws.topk_idx, h->rws.topk_w, h->dws, yd,
                                                      h->rws.err, h->sms, s, false, &h->wq))))
        return st;
      if ((st = prof_mark(h, s, 2))) return st;
      return prof_finish_call(h, s, 3);
    }
    if ((st = cuda_status(moe::launch_decode_q4_gateup(xd, h->wq, h->D, h->rws.topk_idx,
                                                       h->rws.topk_w, h->dws, h->sms, s))))
      return st;
    if ((st = prof_mark(h, s, 2))) return st;
    if ((st = cuda_status(moe::launch_decode_q4_down_combine(h->wq, h->D, h->dws, yd, h->sms,
                                                             s))))
      return st;
    return prof_finish_call(h, s, 3);
  }

  if (use_gemv(h, T) || per_token(h, T)) {
    const moe::DecodeWeights W = decode_weights(h);
    for (int t = 0; t < T; ++t) {
      const __nv_bfloat16* xt = xd + (size_t)t * h->D.d;
      if ((st = prof_mark(h, s, 3 * t))) return st;
      // the router alone: the shared expert's gate/up runs in the gate/up launch
      if ((st = cuda_status(moe::launch_decode_router_shared(xt, W, h->D, nullptr, nullptr,
                                                             nullptr, nullptr, h->dws,
                                                             h->rws.err, s, false))))
        return st;
      if ((st = prof_mark(h, s, 3 * t + 1))) return st;
      __nv_bfloat16* yt = yd + (size_t)t * h->D.d;
      if (moe::decode_stream_fits(h->D, h->sms)) {
        // selection, gate/up and down with the combine in one launch (its profiling slot 2
        // stays empty)
        const bool expire = h->expire_calls > 0;
        if (expire) --h->expire_calls;
        if ((st = cuda_status(moe::launch_decode_stream(xt, W, h->D, h->rws.topk_idx,
                                                        h->rws.topk_w, h->dws, yt, h->rws.err,
                                                        h->sms, s, expire))))
          return st;
        if ((st = prof_mark(h, s, 3 * t + 2))) return st;
        continue;
      }
      if ((st = cuda_status(moe::launch_decode_gateup(xt, W, h->D, h->rws.topk_idx,
                                                      h->rws.topk_w, h->dws, s))))
        return st;
      if ((st = prof_mark(h, s, 3 * t + 2))) return st;
      if ((st = cuda_status(moe::launch_decode_down_combine(W, h->D, h->dws, yt, s))))
        return st;
    }
    return prof_finish_call(h, s, 3 * T);
  }

  if (!h->q4 && use_batch(h, T)) {  // the small-batch matrix-vector path reads bf16
    const moe::DecodeWeights W = decode_weights(h);
    if ((st = prof_mark(h, s, 0))) return st;
    if ((st = cuda_status(moe::launch_decode_batch_router_shared(xd, W, h->D, T, nullptr, nullptr,
                                                                 nullptr, nullptr, h->dws, s,
                                                                 true))))
      return st;
    if ((st = prof_mark(h, s, 1))) return st;
    if ((st = cuda_status(moe::launch_decode_batch_gateup(xd, W, h->D, T, h->rws.topk_idx,
                                                          h->rws.topk_w, h->dws, h->sms, s))))
      return st;
    if ((st = prof_mark(h, s, 2))) return st;
    if ((st = cuda_status(moe::launch_decode_batch_down_combine(W, h->D, T, h->dws, yd, h->sms,
                                                                s))))
      return st;
    return prof_finish_call(h, s, 3);
  }

  if (T <= h->Tc) {
    if ((st = forward_gemm(h, xd, T, yd, s, true, small_router(h, T)))) return st;
    return prof_finish_call(h, s, 4);
  }
  // longer than a chunk: the layer over consecutive chunks of at most Tc tokens, in order on
  // the stream (profiled as one entry)
  if ((st = prof_mark(h, s, 0))) return st;
  for (int t0 = 0; t0 < T; t0 += h->Tc) {
    const int n = T - t0 < h->Tc ? T - t0 : h->Tc;
    const size_t off = (size_t)t0 * h->D.d;
    if ((st = forward_gemm(h, xd + off, n, yd + off, s, false, small_router(h, T)))) return st;
  }
  return prof_finish_call(h, s, 1);
}

int moe_forward_host(moe_handle h, const void* x_host, int T, void* y_host, void* stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (T > h->cfg.max_tokens) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!x_host || !y_host) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // y in page-locked host memory that the device can address (and 16-byte aligned): the
  // layer's last kernel writes it in place over the host link, so no device-to-host copy
  // follows; any other y goes through the staging buffer and a copy
  char* y_dev = static_cast<char*>(device_view(y_host));
  // x likewise: the SMs copy it into the staging buffer (faster over the host link than the
  // copy engine); any other x is copied by cudaMemcpyAsync
  const char* x_dev = static_cast<const char*>(device_view(x_host));
  // through the staging buffers one chunk at a time (stream order keeps the reuse safe)
  const char* xb = static_cast<const char*>(x_host);
  char* yb = static_cast<char*>(y_host);
  for (int t0 = 0; t0 < T; t0 += h->Tc) {
    const int n = T - t0 < h->Tc ? T - t0 : h->Tc;
    const size_t off = (size_t)t0 * h->D.d * 2, bytes = (size_t)n * h->D.d * 2;
    int st = x_dev && bytes % 16 == 0
                 ? cuda_status(moe::launch_host_copy(x_dev + off, h->x_stage, bytes, h->sms, s))
                 : cuda_status(cudaMemcpyAsync(h->x_stage, xb + off, bytes,
                                               cudaMemcpyHostToDevice, s));
    if (st) return st;
    if (y_dev) {
      if ((st = moe_forward(h, h->x_stage, n, y_dev + off, stream))) return st;
      continue;
    }
    if ((st = moe_forward(h, h->x_stage, n, h->y_stage, stream))) return st;
    if ((st = cuda_status(cudaMemcpyAsync(yb + off, h->y_stage, bytes, cudaMemcpyDeviceToHost, s))))
      return st;
  }
  return MOE_OK;
}

int moe_get_device_error(moe_handle h, void* stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  int st = cuda_status(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  if (st) return st;
  int v = 0;
  if ((st = cuda_status(cudaMemcpy(&v, h->rws.err, sizeof(int), cudaMemcpyDeviceToHost))))
    return st;
  if (v != 0 && (st = cuda_status(cudaMemset(h->rws.err, 0, sizeof(int))))) return st;
  return v;
}

namespace {
void prof_release(moe_handle h) {
  for (cudaEvent_t e : h->prof_ev) cudaEventDestroy(e);
  h->prof_ev.clear();
  h->prof_calls = h->prof_done = h->prof_nk = 0;
}
}  // namespace

int moe_profile_begin(moe_handle h, int n_calls) {
  if (!h || n_calls < 1 || n_calls > 1024) return MOE_ERR_INVALID_ARG;
  prof_release(h);
  const size_t n = (size_t)n_calls * (moe_handle_s::kMaxKernels + 1);
  h->prof_ev.reserve(n);
  for (size_t i = 0; i < n; ++i) {
    cudaEvent_t e;
    int st = cuda_status(cudaEventCreate(&e));
    if (st) {
      prof_release(h);
      return st;
    }
    h->prof_ev.push_back(e);
  }
  h->prof_calls = n_calls;
  return MOE_OK;
}

int moe_profile_end(moe_handle h, float* ms, int capacity, int* n_kernels, int* n_calls) {
  if (!h || !ms || capacity < 0 || !n_kernels || !n_calls) return MOE_ERR_INVALID_ARG;
  const int nk = h->prof_nk, done = h->prof_done, stride = moe_handle_s::kMaxKernels + 1;
  for (int i = 0; i < capacity; ++i) ms[i] = 0.f;
  int st = MOE_OK;
  for (int c = 0; c < done && st == MOE_OK; ++c) {
    for (int i = 0; i < nk && i < capacity; ++i) {
      float t = 0.f;
      st = cuda_status(cudaEventSynchronize(h->prof_ev[(size_t)c * stride + i + 1]));
      if (st) break;
      st = cuda_status(cudaEventElapsedTime(&t, h->prof_ev[(size_t)c * stride + i],
                                            h->prof_ev[(size_t)c * stride + i + 1]));
      if (st) break;
      ms[i] += t;
    }
  }
  *n_kernels = nk;
  *n_calls = done;
  prof_release(h);
  return st;
}

int moe_test_expire_waits(moe_handle h, int n_calls) {
  if (!h || n_calls < 0) return MOE_ERR_INVALID_ARG;
  if (h->q4 || !moe::decode_stream_fits(h->D, h->sms)) return MOE_ERR_UNSUPPORTED;
  h->expire_calls = n_calls;
  return MOE_OK;
}

int moe_destroy(moe_handle h) {
  if (!h) return MOE_OK;
  prof_release(h);
  int st = MOE_OK;
  if (h->ws) st = cuda_status(cudaFree(h->ws));
  delete h;
  return st;
}

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration or size";
    case MOE_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case MOE_ERR_CUDA: return "CUDA call failed";
    case MOE_ERR_TIMEOUT: return "a kernel's bounded wait expired";
    case MOE_ERR_DEVICE: return "kernel detected an inconsistent state";
    case MOE_ERR_NO_MEMORY: return "out of memory";
    default: return "unknown status";
  }
}

int moe_last_cuda_error(void) { return g_last_cuda_error; }

}  // extern "C"
