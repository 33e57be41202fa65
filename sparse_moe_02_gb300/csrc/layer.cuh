// Internal interface between the C ABI (api.cu) and the kernel files: sizes, the
// routing-workspace layout, kernel argument blocks and launcher declarations.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

constexpr int kE = 256;            // experts
constexpr int kTopK = 8;           // kept per token
constexpr int kBlockTokens = 128;  // tokens per router / scatter block (the MMA M)
constexpr int kChunkRows = 192;    // most token rows in one grouped-GEMM work unit (MMA N)
constexpr int kRowAlign = 16;      // expert groups start on 16-row boundaries (MMA N step)
constexpr int kMTile = 128;        // weight rows per work unit (MMA M)
constexpr int kBK = 64;            // K elements per pipeline stage (one 128-byte swizzle row)
constexpr int kHBoxRows = 64;      // h rows per TMA box of a down unit (rows past N unused)

__host__ __device__ constexpr int round_up(int v, int m) { return (v + m - 1) / m * m; }

// One grouped-GEMM work unit: expert group g (g == kE: the shared expert), first padded row
// p0, valid rows nrows (<= kChunkRows), weight row tile mt, and cid, the index of its chunk
// (group, rows) -- the down units of a chunk wait for all gate/up units of the same chunk.
struct Unit {
  int g, p0, nrows, mt, cid;
};

// Device workspace of the routing chain (all sized for max_tokens at create time).
struct RouteWs {
  int32_t* topk_idx;  // [T][8] when the caller does not supply one
  float* topk_w;      // [T][8]
  int32_t* hist;      // [nblk][E] assignments per (token block, expert)
  int32_t* blkpre;    // [nblk][E] assignments of earlier blocks, per expert (two-launch plan)
  int32_t* offsets;   // [E+1]
  int32_t* poff;      // [E+2] padded start row of each group (E = shared), poff[E+1] = total
  int32_t* perm;      // [T*8] slot -> t*8+j
  int32_t* prow;      // [T][9] padded row of (t, j); column 8 = the shared expert's row
  int32_t* grow;      // [P] token of each padded row (0 for padding rows)
  Unit* units_gu;     // gate/up work units
  Unit* units_dn;     // down work units
  int32_t* n_units;   // [2]: gate/up, down
  int32_t* next_unit; // dynamic schedule counter of the expert kernel (zeroed by the plan)
  int32_t* chunk_done;  // [chunks] gate/up units finished per chunk (zeroed by the plan)
  int* err;           // device error word
};

struct Dims {
  int d, f, fs, hdim;  // hdim = max(f, fs): row pitch of the h buffer
};

// Launch with programmatic dependent launch allowed: the kernel may start while its
// predecessor on the stream finishes; every kernel here calls griddepcontrol.wait before it
// touches memory that earlier work on the stream writes.
template <typename K, typename... Args>
inline cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Sets the dynamic shared-memory limits of the kernels that need more than 48 KB.
cudaError_t prepare_route_kernels();
cudaError_t prepare_expert_kernels();
cudaError_t prepare_decode_kernels(int hdim);

// ---------------------------------------------------------------- launchers (stream-ordered)

// Router GEMM + top-8 + softmax + per-block histogram (tensor cores), one block per 128 tokens.
cudaError_t launch_router_topk(const CUtensorMap& tm_x, const CUtensorMap& tm_wr,
                               const float* bias, int T, const Dims& D, int32_t* topk_idx,
                               float* topk_w, const RouteWs& ws, cudaStream_t s);

// Per-expert totals, offsets, padded group starts, the work-unit lists and the counting-sort
// scatter (perm, prow, grow): one launch of one block per token block while there are at most
// kFusedPlanBlocks token blocks, else a one-block plan launch and a scatter launch.
constexpr int kFusedPlanBlocks = 128;
cudaError_t launch_route_plan_scatter(int T, const Dims& D, const int32_t* topk_idx,
                                      int32_t* perm, const RouteWs& ws, cudaStream_t s);

struct Q4Weights;

// Copy of `bytes` (a multiple of 16; both pointers 16-byte aligned) from page-locked host memory
// the device can address to device memory, by the SMs (at most 4 blocks per SM).
cudaError_t launch_host_copy(const void* src, void* dst, size_t bytes, int sms, cudaStream_t s);

// Both grouped GEMMs in one persistent launch: the gate/up units (SwiGLU epilogue, h [P][hdim]
// bf16) and then the down units (ys [P][d] bf16), a down unit starting once every gate/up unit
// of its chunk has published its h.  With q4 NULL the weight maps are bf16 maps (box 64 x
// 128, 128-byte swizzle); with q4 set they are maps of the 4-bit code bytes (box 32 bytes x
// 128 rows, no swizzle) and q4 supplies the scales and biases.
cudaError_t launch_experts(const __nv_bfloat16* x, const CUtensorMap& tm_wg,
                           const CUtensorMap& tm_wu, const CUtensorMap& tm_wsg,
                           const CUtensorMap& tm_wsu, const CUtensorMap& tm_h,
                           const CUtensorMap& tm_wd, const CUtensorMap& tm_wsd, const Dims& D,
                           const RouteWs& ws, __nv_bfloat16* h, __nv_bfloat16* ys, int grid,
                           cudaStream_t s, const Q4Weights* q4 = nullptr);

// y[t] = sum_j w[t][j] ys[prow[t][j]] + ys[prow[t][8]] in fp32, rounded once to bf16
// (persistent: at most `grid` blocks, one per SM).
cudaError_t launch_combine(int T, const Dims& D, const float* topk_w, const RouteWs& ws,
                           const __nv_bfloat16* ys, __nv_bfloat16* y, int grid, cudaStream_t s);

// ---------------------------------------------------------------- batch-1 decode path

// ---------------------------------------------------------------- 4-bit weights

// One row of a 4-bit group-affine matrix: codes (K/2 bytes, two codes per byte, the lower
// nibble first), scales and biases (K/64 bf16, one per group of 64 inputs).
struct Q4Row {
  const uint8_t* codes;
  const __nv_bfloat16* scales;
  const __nv_bfloat16* biases;
};

// A whole matrix of rows of K inputs (row r at codes + r K/2, scales/biases + r K/64).
struct Q4Matrix {
  const uint8_t* codes;
  const __nv_bfloat16* scales;
  const __nv_bfloat16* biases;
  __host__ __device__ Q4Row row(size_t r, int K) const {
    return Q4Row{codes + r * (size_t)(K / 2), scales + r * (size_t)(K / 64),
                 biases + r * (size_t)(K / 64)};
  }
};

struct Q4Weights {
  const __nv_bfloat16* w_r;  // the router stays bf16
  const float* bias;
  Q4Matrix gate, up, down, s_gate, s_up, s_down;
};

// Small-batch decode (2..kGemvMaxTokens tokens): shapes whose per-block copies of x
// (T d bf16) and h (T 9 hdim fp32) fit in shared memory.
constexpr int kGemvMaxTokens = 8;
constexpr int kBatchMaxTHdim = 4096;  // T * max(f, fs)
constexpr int kBatchMaxTD = 65536;    // T * d

struct DecodeWs {
  float* logits;   // [kGemvMaxTokens][E]
  int* counter;    // last-block detection of the router
  int* gu_next;    // grid barrier counter of the streamed launch (zeroed by the router launch)
  float* hdec;     // [kGemvMaxTokens][9][hdim] fp32: routed experts j = 0..7, shared = 8
};

struct DecodeWeights {
  const __nv_bfloat16 *w_r, *w_gate, *w_up, *w_down, *ws_gate, *ws_up, *ws_down;
  const float* bias;
};

// Streamed batch-1 decode: after the router launch (routing only), one launch of one block per
// SM that selects, streams the shared expert's and the 8 selected experts' gate/up rows (h into
// dw.hdec), meets at a grid-wide barrier (counter dw.gu_next, zeroed by the router launch) and
// combines its slice of outputs from the down rows it copied meanwhile; block 0 writes
// topk_idx / topk_w.  Shapes whose buffers exceed these limits use the per-warp kernels
// (launch_decode_gateup, launch_decode_down_combine).
constexpr int kStreamMaxD = 2048;
constexpr int kStreamMaxSmem = 218 * 1024;  // leaves room for a router block on the same SM
bool decode_stream_fits(const Dims& D, int sms, bool q4 = false);
cudaError_t prepare_decode_stream_kernels();
// expire: the launch's grid barrier waits for one arrival more than there are blocks, for
// 1 ms, then records MOE_ERR_TIMEOUT and the blocks leave without combining (the test of the
// timeout path).
// moe_check_routing's kernel (check.cu): sets *status to the device-state error if the routing
// (topk_idx [T][8], offsets [E+1], perm [8T]) is inconsistent; leaves it unchanged otherwise.
cudaError_t launch_check_routing(const int32_t* topk_idx, const int32_t* offsets,
                                 const int32_t* perm, int T, int* status, cudaStream_t s);

cudaError_t launch_decode_stream(const __nv_bfloat16* x, const DecodeWeights& W, const Dims& D,
                                 int32_t* topk_idx, float* topk_w, const DecodeWs& dw,
                                 __nv_bfloat16* y, int* err, int sms, cudaStream_t s,
                                 bool expire = false, const Q4Weights* q4 = nullptr);

// Router GEMV (logits) and the shared expert's gate/up GEMV, one launch.  When topk_idx is
// not NULL (routing requested) the last router block to finish also writes the top 8.
cudaError_t launch_decode_router_shared(const __nv_bfloat16* x, const DecodeWeights& W,
                                        const Dims& D, int32_t* topk_idx, float* topk_w,
                                        int32_t* offsets, int32_t* perm, const DecodeWs& dw,
                                        int* err, cudaStream_t s, bool with_shared);

// Top-8 selection from the logits and the gate/up GEMV of the 8 selected experts with the
// SwiGLU fused; block 0 writes the selection to topk_idx / topk_w.
cudaError_t launch_decode_gateup(const __nv_bfloat16* x, const DecodeWeights& W, const Dims& D,
                                 int32_t* topk_idx, float* topk_w, const DecodeWs& dw,
                                 cudaStream_t s);

// Down GEMV of the 8 experts and the shared expert, weighted and combined in fixed order.
cudaError_t launch_decode_down_combine(const DecodeWeights& W, const Dims& D, const DecodeWs& dw,
                                       __nv_bfloat16* y, cudaStream_t s);

// Small-batch decode of T = 2..kGemvMaxTokens tokens (decode_batch_fits): the same three
// launches as the single-token path, over the union of the tokens' experts (each weight row
// read once, applied to every token that chose it).  With topk_idx not NULL the router launch
// is routing only (its last block writes topk_idx, topk_w and, where not NULL, offsets and
// perm); with plan not NULL it is the routing of the tensor-core schedule for T <= 128: the
// last block also writes the plan (offsets, group starts, unit lists, chunk counters) into
// *plan and scatters the tokens (perm, the padded rows), so no plan launch follows.
bool decode_batch_fits(const Dims& D, int T);
cudaError_t prepare_decode_batch_kernels();
cudaError_t launch_decode_batch_router_shared(const __nv_bfloat16* x, const DecodeWeights& W,
                                              const Dims& D, int T, int32_t* topk_idx,
                                              float* topk_w, int32_t* offsets, int32_t* perm,
                                              const DecodeWs& dw, cudaStream_t s,
                                              bool with_shared, const RouteWs* plan = nullptr);
cudaError_t launch_decode_batch_gateup(const __nv_bfloat16* x, const DecodeWeights& W,
                                       const Dims& D, int T, int32_t* topk_idx, float* topk_w,
                                       const DecodeWs& dw, int sms, cudaStream_t s);
cudaError_t launch_decode_batch_down_combine(const DecodeWeights& W, const Dims& D, int T,
                                             const DecodeWs& dw, __nv_bfloat16* y, int sms,
                                             cudaStream_t s);

// Batch-1 decode with 4-bit experts: the router launch of the bf16 path (the router stays
// bf16), then the shared expert's and the 8 selected experts' 4-bit gate/up, and the down rows
// weighted and combined in fixed order.
cudaError_t prepare_decode_q4_kernels();
cudaError_t launch_decode_q4_gateup(const __nv_bfloat16* x, const Q4Weights& W, const Dims& D,
                                    int32_t* topk_idx, float* topk_w, const DecodeWs& dw,
                                    int sms, cudaStream_t s);
cudaError_t launch_decode_q4_down_combine(const Q4Weights& W, const Dims& D, const DecodeWs& dw,
                                          __nv_bfloat16* y, int sms, cudaStream_t s);

}  // namespace moe
