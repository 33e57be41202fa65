/*
 * Gated DeltaNet recurrent scan on one GB300 GPU (sm_103a), part of libmoe.
 *
 * Source: "Optimizing on-device inference for Apple Silicon", § "Keep recurrent state on chip":
 * during prefill a Gated DeltaNet layer scans the prompt in token order while carrying a
 * recurrent state forward; the state is a matrix; the optimised kernel gives each of its
 * columns to one group of SIMD lanes, which loads the column into registers once, carries it
 * through the whole scan, exchanges partial results with cross-lane operations rather than
 * shared memory, and writes the finished state back once; the state and its gate are 32-bit
 * floats (rounding errors add up over the sequential updates), the query and key bf16.
 *
 * The update rule is not printed there; this library takes the gated delta rule (Yang, Kautz &
 * Hatamizadeh, "Gated Delta Networks: Improving Mamba2 with Delta Rule"), per head and token t,
 * with the state S stored key-major (S[i][j], i < dk a key coordinate, j < dv a value one):
 *
 *   S_t = alpha_t S_{t-1} + beta_t k_t (v_t - alpha_t S_{t-1}^T k_t)^T
 *       = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
 *   o_t = S_t^T q_t
 *
 * Each value column j of S evolves on its own (its update needs only column j and the token's
 * k, q, v[j] and gates), which is what lets one lane group own one column.
 *
 * Data types and layouts (row-major; "bf16" = IEEE bfloat16 bits):
 *   q, k      [T][H][dk] bf16 (normalisation and scaling, if any, are applied by the caller)
 *   v         [T][H][dv] bf16
 *   alpha     [T][H] fp32: the decay gate of each token and head (in (0, 1] for a stable scan)
 *   beta      [T][H] fp32: the write strength (in [0, 1])
 *   state_in  [H][dk][dv] fp32: the state before token 0 (the state a previous prompt chunk
 *             left), or NULL for a zero state
 *   state_out [H][dk][dv] fp32: the state after token T-1; may equal state_in (updated in place)
 *   o         [T][H][dv] bf16: o_t rounded once from fp32
 *
 * Arithmetic: fp32 state and gates; q, k, v widened exactly from bf16.  Per token the kernel
 * forms r_t = S_{t-1}^T k_t and p_t = S_{t-1}^T q_t, then u_t = beta_t (v_t - alpha_t r_t),
 * o_t = alpha_t p_t + (k_t . q_t) u_t (= S_t^T q_t) and S_t = alpha_t S_{t-1} + k_t u_t^T.  Inside
 * each run of 32 tokens (counted from the call's first token) r_t and p_t are taken one token
 * early, as alpha_{t-1} S_{t-2}^T k_t + (k_{t-1} . k_t) u_{t-1} (and likewise with q_t), which
 * is the same value rounded differently.  Sums are fp32 in a fixed order, so a call is
 * deterministic, and a scan split into two calls after a multiple of 32 tokens, the second
 * starting from the first's state_out, gives bit-identical outputs and state (a split elsewhere
 * agrees to rounding).
 *
 * Ownership and threading: every pointer is a device pointer owned by the caller; the call
 * only enqueues one kernel on `stream` (a cudaStream_t as void*, NULL = the legacy default
 * stream) and allocates nothing.  o must not overlap the inputs.
 *
 * Errors (status values of moe.h): MOE_ERR_INVALID_ARG (T < 0, H < 1, a NULL pointer other
 * than state_in; q, k, v, alpha, beta and o may be NULL when T == 0), MOE_ERR_UNSUPPORTED
 * (dk != 128, dv not a multiple of 32 or above 4096, H above 65535), MOE_ERR_ALIGNMENT (q, k, v, o
 * not 16-byte aligned; alpha, beta not 4-byte aligned; state_in, state_out not 8-byte aligned),
 * MOE_ERR_CUDA (the launch failed).  The kernel has no waits that can time out.
 */
#ifndef GDN_H
#define GDN_H

#include <stdint.h>

#include "moe.h"

#ifdef __cplusplus
extern "C" {
#endif

int gdn_scan(const void* q, const void* k, const void* v, const float* alpha, const float* beta,
             const float* state_in, float* state_out, void* o, int64_t T, int H, int dk, int dv,
             void* stream);

#ifdef __cplusplus
}
#endif

#endif
