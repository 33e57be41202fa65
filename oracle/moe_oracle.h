/*
 * CPU oracle of the mixture-of-experts FFN layer.  TEST INFRASTRUCTURE ONLY: the tests, the
 * smoke check and the CPU-baseline timing call it; the product library never does.
 *
 * It is the plain definition of what the layer computes, written out as slow loops in fp32
 * over bf16 inputs (each input widened exactly), and it shares no code with the CUDA path.
 *
 * Sources ("Optimizing on-device inference for Apple Silicon"):
 *   - § "three distinct workload shapes": a router scores 256 experts per token, keeps eight,
 *     and a shared expert processes every token.
 *   - § "Keep expert routing on the GPU": histogram of assignments per expert, prefix scan
 *     into start offsets, scatter of rows into expert groups.
 *   - § "Dequantize weights during matrix multiplication": fp32 accumulation, bf16 output.
 *   - § "Reduce intermediate and state traffic": the two expert input projections with
 *     their gated activation; the output projection with its routing score and the shared
 *     expert's result.
 * Readings where the page is silent: softmax over the kept logits, SwiGLU (silu(gate)*up),
 * shared expert ungated with weight 1, combine in ascending expert id then the shared
 * expert, one final bf16 rounding; ties in selection go to the lower expert id.
 *
 * Layouts (row-major, bf16 passed as uint16 bits; weights output-major):
 *   x [T][d]; w_r [E][d]; bias [E] fp32 or NULL; per expert e: w_gate[e], w_up[e] [f][d],
 *   w_down[e] [d][f]; shared: ws_gate, ws_up [fs][d], ws_down [d][fs].
 * All functions return 0 on success and a negative value on invalid arguments.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int d, E, k, f, fs;
} oracle_dims;

/* Router logits in fp64 from the exact bf16 inputs, bias added in fp64.  Used to measure the
 * gap between the k-th and (k+1)-th largest logit when inputs are drawn. */
int oracle_router_logits_f64(const uint16_t* x, int64_t T, int d, const uint16_t* w_r, int E,
                             const float* bias, double* logits, int nthreads);

/* Router logits in fp32: sum over i ascending of x[t][i]*w_r[e][i], then + bias[e]. */
int oracle_router_logits_f32(const uint16_t* x, int64_t T, int d, const uint16_t* w_r, int E,
                             const float* bias, float* logits, int nthreads);

/* Keep the k largest of each row of logits [T][E] (ties: lower expert id first), stored in
 * ascending expert id; weights = softmax over the kept logits, aligned with the ids. */
int oracle_select(const float* logits, int64_t T, int E, int k, int32_t* topk_idx,
                  float* topk_w);

/* Counting sort of the T*k assignments by expert: counts[E], offsets[E+1] (exclusive scan,
 * offsets[E] = T*k), perm[T*k] (slot -> t*k+j, experts ascending, tokens ascending within an
 * expert) and inv_perm[T*k] ((t,j) -> slot). */
int oracle_route_structure(const int32_t* topk_idx, int64_t T, int E, int k, int32_t* counts,
                           int32_t* offsets, int32_t* perm, int32_t* inv_perm);

/* One SwiGLU expert on one row: h[f] (fp32, unrounded) and o[d] (fp32). */
int oracle_expert_ffn(const uint16_t* x_row, int d, const uint16_t* w_gate, const uint16_t* w_up,
                      const uint16_t* w_down, int f, float* h, float* o);

/* The layer's output rows for the listed tokens (tokens == NULL: all T tokens in order).
 * w_gate/w_up/w_down are arrays of E pointers; an expert that no listed token selects may be
 * NULL.  y [n_tokens][d] bf16; topk_idx/topk_w [n_tokens][k] may be NULL. */
int oracle_forward(const oracle_dims* D, const uint16_t* x, int64_t T, const uint16_t* w_r,
                   const float* bias, const uint16_t* const* w_gate, const uint16_t* const* w_up,
                   const uint16_t* const* w_down, const uint16_t* ws_gate, const uint16_t* ws_up,
                   const uint16_t* ws_down, const int64_t* tokens, int64_t n_tokens, uint16_t* y,
                   int32_t* topk_idx, float* topk_w, int nthreads);

/* 4-bit group-affine matrix with rows of K inputs (K a multiple of 64): codes [rows][K/2]
 * (two 4-bit codes per byte, the lower nibble first), scales and biases [rows][K/64] bf16.
 * Weight (r, i) = scales[r][i/64] * q + biases[r][i/64] in fp32 (one multiply, one add), q the
 * code of input i (§ "Dequantize weights during matrix multiplication": 4-bit weights in
 * groups with a scale and a bias). */
typedef struct {
  const uint8_t* codes;
  const uint16_t* scales;
  const uint16_t* biases;
} oracle_q4;

/* The dequantized fp32 weights of a 4-bit matrix, out [rows][K]. */
int oracle_dequant_q4(const oracle_q4* m, int64_t rows, int K, float* out);

/* oracle_forward with 4-bit experts: w_gate/w_up/w_down are arrays of E matrices (codes NULL
 * for an expert no listed token selects); the router stays bf16. */
int oracle_forward_q4(const oracle_dims* D, const uint16_t* x, int64_t T, const uint16_t* w_r,
                      const float* bias, const oracle_q4* w_gate, const oracle_q4* w_up,
                      const oracle_q4* w_down, const oracle_q4* ws_gate, const oracle_q4* ws_up,
                      const oracle_q4* ws_down, const int64_t* tokens, int64_t n_tokens,
                      uint16_t* y, int32_t* topk_idx, float* topk_w, int nthreads);

#ifdef __cplusplus
}
#endif

#endif
