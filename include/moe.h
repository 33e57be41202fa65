/*
 * libmoe -- one mixture-of-experts FFN layer on one GB300 GPU (sm_103a), behind a C ABI.
 *
 * What the layer computes (source: "Optimizing on-device inference for Apple Silicon"):
 *   - § "three distinct workload shapes": a router scores E = 256 experts per token and keeps
 *     eight; a shared expert processes every token; experts receive uneven token counts.
 *   - § "Keep expert routing on the GPU": after selection, a histogram counts the
 *     assignments of each expert, a prefix scan turns counts into start offsets, a scatter
 *     places rows in their expert groups, and a block map lists the fixed-size blocks the
 *     grouped GEMM processes -- all on the GPU, with no CPU-GPU synchronisation in the layer.
 *   - § "Match tile size to expert load": the grouped GEMM's tile fits the rows an expert has.
 *   - § "Dequantize weights during matrix multiplication": fp32 accumulation, bf16 output.
 *   - § "Optimize the one-row weight path" and § "Reduce intermediate and state traffic":
 *     batch-1 decode is a matrix-vector product; the two expert input projections are fused
 *     with their gated activation, and the output projection with its routing score and the
 *     shared expert's result.
 * Readings where the page is silent (fixed by this library):
 *   logits[t][e] = x[t] . w_router[e] (+ router_bias[e]); the k = 8 largest are kept (ties to
 *   the lower expert id) and listed in ascending expert id; their weights are the softmax
 *   over the kept logits; every expert (and the shared expert) is a SwiGLU FFN
 *   o = W_down (silu(W_gate x) * (W_up x)) with silu(g) = g / (1 + e^-g); the shared expert
 *   is ungated with weight 1;  y[t] = sum_j w[t][j] o_{e_j}(x[t]) + o_shared(x[t]),
 *   accumulated in fp32 in ascending expert id and then the shared expert, rounded once
 *   to bf16.
 *
 * Data types and layouts (row-major; "bf16" = IEEE bfloat16 bits, 2 bytes):
 *   x [T][d] bf16, y [T][d] bf16.
 *   w_router [E][d] bf16 (the d x E router matrix stored transposed, input dim contiguous).
 *   w_gate, w_up [E][f][d] bf16; w_down [E][d][f] bf16: every weight is output-major with the
 *   input dimension contiguous, like a linear layer's weight matrix.
 *   ws_gate, ws_up [fs][d] bf16; ws_down [d][fs] bf16 (shared expert).
 *   router_bias [E] fp32 or NULL.
 *
 * Ownership and threading:
 *   - Weights are BORROWED device pointers: the caller keeps them alive and unchanged for the
 *     lifetime of the handle; nothing is copied.
 *   - The handle owns its device workspace, sized for cfg.max_tokens at moe_create.
 *   - x, y and the routing outputs are owned by the caller.
 *   - moe_route / moe_forward / moe_forward_host only enqueue work on the given stream (a
 *     cudaStream_t passed as void*, NULL = the legacy default stream) and return; they never
 *     synchronise with the host.  A handle must be used on one stream at a time.
 *   - All device pointers must be 16-byte aligned; y must not overlap x.
 *
 * Errors: every call returns a moe_status.  Invalid arguments are rejected before anything is
 * enqueued.  Kernels never trap: a device-side failure (a bounded wait that timed out) is
 * recorded in a device error word that moe_get_device_error reads and clears.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* NULL handle/pointer, T < 0, bad config value */
  MOE_ERR_UNSUPPORTED = 2, /* E != 256, k != 8, d/f/fs not a multiple of 128 or out of range,
                              T > max_tokens */
  MOE_ERR_ALIGNMENT = 3,   /* a device pointer is not 16-byte aligned */
  MOE_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed (see moe_last_cuda_error) */
  MOE_ERR_TIMEOUT = 5,     /* a kernel's bounded wait expired (device error word) */
  MOE_ERR_DEVICE = 6,      /* a kernel detected an inconsistent internal state */
  MOE_ERR_NO_MEMORY = 7    /* workspace allocation failed */
} moe_status;

/* Kernel schedule: AUTO uses the matrix-vector path when T == 1 (with bf16 experts also when
 * T == 2, once per token) and the tensor-core grouped-GEMM path otherwise.  GEMM forces the
 * tensor-core path.  GEMV forces the matrix-vector path: T == 1, or 2 <= T <= 8 when the
 * shape fits (T * max(f, fs) <= 4096 and T * d <= 65536), where every weight row of the union
 * of the tokens' experts is read once and applied to each token that chose it (§ "Limits of
 * further optimization": verifying a few draft tokens at once); other T are rejected with
 * MOE_ERR_UNSUPPORTED. */
typedef enum { MOE_SCHEDULE_AUTO = 0, MOE_SCHEDULE_GEMM = 1, MOE_SCHEDULE_GEMV = 2 } moe_schedule;

typedef struct moe_handle_s* moe_handle;

typedef struct {
  int d;              /* hidden size: multiple of 128, 128 <= d <= 8192 */
  int n_experts;      /* E: must be 256 */
  int top_k;          /* k: must be 8 */
  int ffn_dim;        /* f, routed expert inner dim: multiple of 128, 128 <= f <= 2048 */
  int shared_ffn_dim; /* fs, shared expert inner dim: multiple of 128, 128 <= fs <= 2048 */
  int max_tokens;     /* largest T accepted later: 1 <= max_tokens <= 1048576 */
  int schedule;       /* a moe_schedule value */
  int chunk_tokens;   /* 0, or 1 <= chunk_tokens: moe_forward / moe_forward_host run the layer
                         over at most this many tokens at a time (§ "Prompt chunking": long
                         prompts in bounded pieces), so the per-slot expert buffers (about
                         9 T (2 d + 2 max(f, fs)) bytes) are sized for a chunk, not for
                         max_tokens.  Tokens are independent: the output is byte-identical to
                         the unchunked layer.  moe_route is never chunked. */
} moe_config;

typedef struct {           /* device pointers, borrowed (see above) */
  const void* w_router;    /* bf16 [E][d] */
  const float* router_bias;/* fp32 [E], or NULL for no bias */
  const void* w_gate;      /* bf16 [E][f][d] */
  const void* w_up;        /* bf16 [E][f][d] */
  const void* w_down;      /* bf16 [E][d][f] */
  const void* ws_gate;     /* bf16 [fs][d] */
  const void* ws_up;       /* bf16 [fs][d] */
  const void* ws_down;     /* bf16 [d][fs] */
} moe_weights;

/* Validates cfg and w, allocates the workspace on the current CUDA device, prepares the
 * kernels, and returns a handle in *out.  May synchronise the device.  On failure *out is
 * NULL and nothing stays allocated. */
int moe_create(const moe_config* cfg, const moe_weights* w, moe_handle* out);

/* 4-bit group-affine matrix (§ "Dequantize weights during matrix multiplication": weights in
 * 4 bits, in groups of 64 inputs with a scale and a bias, dequantized inside the matrix
 * kernel).  Rows of K inputs (K a multiple of 128); weight (r, i) = scales[r][i/64] * q +
 * biases[r][i/64], q = the 4-bit code of input i.  Device pointers, borrowed like the bf16
 * weights, each 16-byte aligned. */
typedef struct {
  const void* codes;  /* uint8 [rows][K/2]: two codes per byte, input 2i in the lower nibble */
  const void* scales; /* bf16 [rows][K/64] */
  const void* biases; /* bf16 [rows][K/64] */
} moe_q4_matrix;

typedef struct {
  const void* w_router;     /* bf16 [E][d]: the router stays bf16 */
  const float* router_bias; /* fp32 [E], or NULL */
  moe_q4_matrix w_gate;     /* E*f rows of d inputs */
  moe_q4_matrix w_up;       /* E*f rows of d inputs */
  moe_q4_matrix w_down;     /* E*d rows of f inputs */
  moe_q4_matrix ws_gate;    /* fs rows of d inputs */
  moe_q4_matrix ws_up;      /* fs rows of d inputs */
  moe_q4_matrix ws_down;    /* d rows of fs inputs */
} moe_weights_q4;

/* moe_create for 4-bit experts.  T == 1 under AUTO or GEMV runs the batch-1 matrix-vector
 * path on the codes; every other T (and T == 1 under GEMM) runs the tensor-core path, whose
 * grouped GEMM dequantizes each 64-input step of a weight tile to bf16 (scale * q + bias,
 * rounded once) inside the kernel.  The small-batch matrix-vector path reads bf16 experts
 * only: under GEMV, moe_forward and moe_route with T > 1 return MOE_ERR_UNSUPPORTED. */
int moe_create_q4(const moe_config* cfg, const moe_weights_q4* w, moe_handle* out);

/* Routing only (§ "Keep expert routing on the GPU"): the same kernels moe_forward runs for
 * this T, so moe_forward's routing equals what this returns.  Device outputs, each may be
 * NULL if not wanted:
 *   topk_idx [T][k] int32  kept experts of each token, ascending expert id;
 *   topk_w   [T][k] fp32   their softmax weights, aligned with topk_idx;
 *   offsets  [E+1] int32   offsets[e] = number of assignments to experts < e, offsets[E]=T*k;
 *   perm     [T*k] int32   slot -> t*k + j: assignments grouped by expert (ascending), tokens
 *                          ascending within a group.
 * T == 0 enqueues nothing and returns MOE_OK. */
int moe_route(moe_handle h, const void* x, int T, int32_t* topk_idx, float* topk_w,
              int32_t* offsets, int32_t* perm, void* stream);

/* Consistency check of a routing as moe_route writes it (device pointers, caller-owned; E = 256,
 * k = 8): topk_idx [T][8] ids in [0, E) and strictly ascending within each token; offsets [E+1]
 * with offsets[0] = 0, non-decreasing, offsets[E] = 8T; perm [8T] such that the slots of group
 * e (offsets[e] <= s < offsets[e+1]) hold entries p = t*8+j with topk_idx[p] = e in strictly
 * ascending order -- which together make perm a permutation whose groups are the experts'
 * histogram in stable token order (§ "Keep expert routing on the GPU").  Enqueues a clear of
 * *status (a device int) and one kernel that sets it to MOE_ERR_DEVICE if any condition fails;
 * read it after the stream has run.  The kernel range-checks every value before using it as an
 * index and reads only within the three arrays' sizes, so arrays in any state give a status,
 * never a fault.  The debug build of the library (libmoe_debug.so, compiled with MOE_DEBUG) runs
 * this check inside every moe_route and every tensor-core forward on the routing it produced,
 * recording MOE_ERR_DEVICE in the handle's device error word (moe_get_device_error).
 * Errors: MOE_ERR_INVALID_ARG (NULL status or offsets, NULL topk_idx/perm with T > 0, T < 0),
 * MOE_ERR_UNSUPPORTED (T > 2^20), MOE_ERR_ALIGNMENT (a pointer not 4-byte aligned),
 * MOE_ERR_CUDA. */
int moe_check_routing(const int32_t* topk_idx, const int32_t* offsets, const int32_t* perm, int T,
                      int* status, void* stream);

/* The layer: y [T][d] bf16 from x [T][d] bf16 (device pointers).  T == 0: no-op. */
int moe_forward(moe_handle h, const void* x, int T, void* y, void* stream);

/* moe_forward on HOST buffers: enqueues the copy of x_host [T][d] (pinned memory for an
 * asynchronous copy) into a handle-owned device buffer and the layer.  When y_host [T][d] is
 * page-locked memory the device can address (cudaHostAlloc / cudaHostRegister, 16-byte
 * aligned), the layer's last kernel writes it in place over the host link; otherwise the result
 * goes to a handle-owned device buffer and is copied into y_host.  The caller synchronises the
 * stream before reading y_host. */
int moe_forward_host(moe_handle h, const void* x_host, int T, void* y_host, void* stream);

/* Synchronises `stream`, then returns and clears the handle's device error word
 * (MOE_OK if no kernel reported a failure since the last call). */
int moe_get_device_error(moe_handle h, void* stream);

/* Test hook for the kernels' bounded waits (failure detection without a GPU fault): the next
 * n_calls batch-1 forwards on this bf16 handle run the streamed decode launch with its grid-wide
 * barrier waiting for one block more than the launch has and giving up after 1 ms.  Each such
 * call leaves y undefined and records MOE_ERR_TIMEOUT in the device error word
 * (moe_get_device_error); its blocks still let their own copies land before they leave, so
 * the next forward runs normally.  MOE_ERR_UNSUPPORTED: a 4-bit handle, or a shape the
 * streamed launch does not take (d > 2048 or too many down rows per block); the calls of
 * other schedules are not affected. */
int moe_test_expire_waits(moe_handle h, int n_calls);

/* Frees the workspace and the handle (synchronises the device).  NULL is accepted. */
int moe_destroy(moe_handle h);

/* Measurement hook: enqueues a read-only stream over bytes (a multiple of 16) of device memory
 * at buf (16-byte aligned) on `stream`; sink is a device word the kernel may write (4-byte
 * aligned).  Time it with events on the stream: a pure read stream can exceed the copy rate
 * of the measured HBM peak, and the benchmark reports it beside the decode roofline. */
int moe_read_probe(const void* buf, size_t bytes, void* sink, void* stream);

/* Static description of a status code. */
const char* moe_status_string(int status);

/* The cudaError_t of the last failed CUDA call made by this library in this thread. */
int moe_last_cuda_error(void);

/* Per-kernel timing, for benchmarks and profilers.  moe_profile_begin(h, n_calls) makes the
 * next n_calls (1..1024) calls of moe_forward record a CUDA event on their stream before each
 * kernel and after the last one (this serialises the kernels of those calls, so the times are
 * per kernel without overlap).  moe_profile_end synchronises on those events, writes to
 * ms[i] the device time of the i-th kernel summed over the recorded calls (i < *n_kernels,
 * at most `capacity` entries), sets *n_calls to the number of calls recorded, and stops
 * profiling.  Kernel order -- tensor-core schedule (4): router_topk, route_plan_scatter (one
 * launch up to T = 16384; above, a plan launch and a scatter launch share this slot),
 * experts (gate/up and down), combine; matrix-vector schedule (3):
 * decode_router_shared, decode_gateup, decode_down_combine (T == 2 under AUTO: those three for
 * each token, 6).  All recorded calls must use one
 * schedule. */
int moe_profile_begin(moe_handle h, int n_calls);
int moe_profile_end(moe_handle h, float* ms, int capacity, int* n_kernels, int* n_calls);

/* Routing of one token without any device allocation.  The pages have no counterpart to
 * this entry point; it exists for callers that cannot call cudaMalloc and so cannot create
 * a handle: a process whose device memory is reserved up front by another allocator (a
 * KV-cache or activation pool owning nearly all of HBM), or latency-critical code that may
 * not call cudaMalloc because it can synchronise the whole device.
 * Computes, for x [d] bf16 (one token) and w_router [E=256][d] bf16 (+ router_bias [E] fp32
 * or NULL), the routing that moe_route computes with T == 1 on a handle: topk_idx [8] int32
 * (the 8 largest logits, ties to the lower id, ascending expert id) and topk_w [8] fp32
 * (their softmax weights), all device pointers owned by the caller.  The logits are fp32 sums
 * of the same products in a different order than the handle's router (for d > 2048 the last
 * bits can differ), so the kept experts are the same whenever the 8th and 9th logits are
 * further apart than fp32 rounding.
 * Scratch: a 1,280-byte file-scope device array (the 256 logits and a block counter) that
 * every GPU loading this library holds until exit.  All calls share it and it keeps the last
 * call's contents: calls that overlap on the GPU race (keep them on one stream or ordered);
 * each call clears the counter before its kernel.  The first call on a device looks up the
 * array's device address (cudaGetSymbolAddress) with that device current; make that first
 * call before any stream capture.  The address is kept per device and context: after a
 * cudaDeviceReset (a new context, where the array may sit elsewhere) the next call looks it
 * up again, so make that call, too, outside any stream capture.  Allocates nothing (no
 * cudaMalloc, cudaFree or allocating library routine).
 * Errors: MOE_ERR_INVALID_ARG (NULL pointer), MOE_ERR_UNSUPPORTED (d not a multiple of 128
 * or outside 128..8192, the limit of its shared-memory copy of x), MOE_ERR_ALIGNMENT (x,
 * w_router not 16-byte aligned; bias, outputs not 4-byte aligned), MOE_ERR_CUDA. */
int moe_route_one_noalloc(const void* x, int d, const void* w_router, const float* router_bias,
                          int32_t* topk_idx, float* topk_w, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
