/*
 * Seeded synthetic inputs for the MoE FFN layer: data only, none of the layer's arithmetic.
 *
 * Both the CPU oracle (through the host functions) and the CUDA library (through the device
 * fill) receive their inputs from this one generator, so the two sides see identical bits.
 *
 * Random words: the splitmix64 sequence (Steele, Lea & Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014): state_i = key + (i+1)*0x9E3779B97F4A7C15, output =
 * the splitmix64 finaliser of state_i.  key = fin(fin(seed) + stream*0x9E3779B97F4A7C15).
 * The sequence is counter-based: any element can be produced on its own.
 *
 * Approximately normal values: Irwin-Hall with 12 terms.  Element i of a stream takes the
 * words 3i, 3i+1, 3i+2, splits them into twelve 16-bit fields b_0..b_11 and forms the
 * integer n = sum(b) - 393210 (= 12*32767.5 rounded so that E[n] = 0).  z = n / 65536 has
 * mean 0 and variance 1 - 2^-32, and is bounded by |z| < 6.  The element is
 * bf16_rne(float(z) * sigma): z is exact in fp32, the product is one IEEE fp32 multiply,
 * then one round-to-nearest-even to bf16, so every machine produces the same bits.
 * (Exact normal samplers need log/cos, whose last bit differs between libraries; the
 * integer Irwin-Hall sum keeps host and device bit-identical.)
 */
#ifndef SYNTH_H
#define SYNTH_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Key of one stream.  stream identifies a tensor, a layer and a redraw round. */
uint64_t synth_key(uint64_t seed, uint64_t stream);

/* Word i of the stream with the given key. */
uint64_t synth_word(uint64_t key, uint64_t i);

/* out[j] = bf16 bits of element (offset + j) of the stream, j < n, scaled by sigma.
 * Splits the work over nthreads host threads (<= 0: one); the result does not depend on it. */
void synth_normal_bf16(uint64_t seed, uint64_t stream, uint64_t offset, uint64_t n,
                       float sigma, uint16_t* out, int nthreads);

/* A uniformly random permutation of 0..n-1 (Fisher-Yates, Knuth vol. 2 Algorithm 3.4.2P,
 * with each index drawn by rejection so that it is exactly uniform). */
void synth_permutation(uint64_t seed, uint64_t stream, int32_t n, int32_t* out);

/* Device fill: the same elements as synth_normal_bf16, written to device memory `dst`
 * (n elements) on the CUDA stream `cuda_stream` (a cudaStream_t, 0 = legacy default).
 * Returns 0 on success or the cudaError_t of the launch. */
int synth_normal_bf16_device(uint64_t seed, uint64_t stream, uint64_t offset, uint64_t n,
                             float sigma, void* dst, void* cuda_stream);

/* 4-bit group-affine weights (groups of 64 along a row's input dimension).
 * Codes: byte j of a stream is byte (j mod 8) of word j/8 (little-endian), two 4-bit codes per
 * byte, the lower nibble first.
 * Scale and bias of group j: u = the top 23 bits of word j, v = 0.75f + float(u) * 2^-24 (one
 * IEEE fp32 add), s = bf16_rne(v * base) (one fp32 multiply, then round to nearest even),
 * bias = -8 s (exact in bf16).  The dequantized weight s*q + bias = s*(q - 8) is centred;
 * base = 0.02 / 4.61 gives it the spread of the bf16 experts' N(0, 0.02). */
void synth_bytes(uint64_t seed, uint64_t stream, uint64_t offset, uint64_t n, uint8_t* out);
void synth_q4_affine(uint64_t seed, uint64_t stream, uint64_t offset, uint64_t n, float base,
                     uint16_t* scales, uint16_t* biases);

/* Uniform fp32 values on [lo, hi): element j is u = float(top 24 bits of word offset + j) * 2^-24
 * (exact), then lo + (hi - lo) * u with one IEEE fp32 subtract, one multiply and one add,
 * each rounded on its own (no fused multiply-add), so every machine produces the same bits. */
void synth_uniform_f32(uint64_t seed, uint64_t stream, uint64_t offset, uint64_t n, float lo,
                       float hi, float* out);

/* Device fills of the same (returns 0 or the cudaError_t of the launch). */
int synth_bytes_device(uint64_t seed, uint64_t stream, uint64_t offset, uint64_t n, void* dst,
                       void* cuda_stream);
int synth_q4_affine_device(uint64_t seed, uint64_t stream, uint64_t offset, uint64_t n,
                           float base, void* scales, void* biases, void* cuda_stream);
int synth_uniform_f32_device(uint64_t seed, uint64_t stream, uint64_t offset, uint64_t n,
                             float lo, float hi, void* dst, void* cuda_stream);

#ifdef __cplusplus
}
#endif

#endif
