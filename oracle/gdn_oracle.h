/*
 * CPU oracle of the Gated DeltaNet recurrent scan.  TEST INFRASTRUCTURE ONLY: the tests, the
 * smoke check and the benchmark's CPU-baseline leg call it; the product library never does.
 *
 * Source: the blog post "Optimizing on-device inference for Apple Silicon", section "Keep
 * recurrent state on chip": during prefill each Gated DeltaNet layer scans the prompt in order
 * and carries a recurrent state forward; the state is a matrix, kept with its gate in 32-bit
 * floating point, while the query and key activations stay bf16; the finished state is written
 * back once, after the scan.  The post does not print the update rule.  This oracle takes the
 * gated delta rule as published (Yang, Kautz & Hatamizadeh, "Gated Delta Networks: Improving
 * Mamba2 with Delta Rule", ICLR 2025), per head and token t, with the state S stored key-major,
 * S[i][j] (i < dk a key coordinate, j < dv a value coordinate), i.e. the transpose of the
 * paper's value-by-key matrix:
 *
 *   decay     S <- alpha_t S
 *   retrieve  r = S^T k_t            (the value the memory currently returns for key k_t)
 *   delta     u = beta_t (v_t - r)   (the error-correcting write of the delta rule)
 *   write     S <- S + k_t u^T
 *   read      o_t = S^T q_t
 *
 * which is S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T, o_t = S_t^T q_t.
 * The gates alpha_t (decay, in (0, 1]) and beta_t (write strength, in [0, 1]) arrive as fp32
 * inputs: the projections and activations that produce them, and q/k normalisation, sit
 * outside the scan.
 *
 * Arithmetic: fp64 throughout over the exactly widened bf16 / fp32 inputs; plain loops in the
 * order above; no FMA contraction.
 */
#ifndef GDN_ORACLE_H
#define GDN_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* q, k [T][H][dk] and v [T][H][dv] bf16 bits; alpha, beta [T][H] fp32; s0 [H][dk][dv] fp32 or
 * NULL (zero state).  Writes o [T][H][dv] and s_out [H][dk][dv] (the state after token T-1) in
 * fp64.  Heads are independent and run on up to nthreads threads; the result does not depend
 * on nthreads.  Returns 0, or -1 on invalid sizes. */
int oracle_gdn_scan(const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* alpha,
                    const float* beta, const float* s0, int64_t T, int H, int dk, int dv,
                    double* o, double* s_out, int nthreads);

#ifdef __cplusplus
}
#endif

#endif
