// 4-bit group-affine arithmetic shared by the batch-1 decode kernels: weight (r, i) =
// scale[r][i / 64] * q + bias[r][i / 64], q the 4-bit code of input i (the lower nibble of a
// byte first).  A row's contribution to a dot product with v is, per piece of 32 inputs,
// scale * sum_i q_i v_i + bias * sum_i v_i, with the sums of v per 32 formed once.
#pragma once

#include "layer.cuh"
#include "ptx.cuh"

namespace moe {

// Vectors in shared memory are stored swizzled: float4 k (k = 0..7) of 32-element piece p sits
// in slot (k + p) mod 8 of the piece, so that eight lanes reading float4 k of eight
// consecutive pieces touch all 32 banks.  Element i -> position:
__host__ __device__ __forceinline__ int swz(int i) {
  return (i & ~31) | ((((i >> 2) + (i >> 5)) & 7) << 2) | (i & 3);
}

// float4 k of piece p of a swizzled vector
__device__ __forceinline__ float4 piece_f4(const float* v, int p, int k) {
  return *reinterpret_cast<const float4*>(v + 32 * p + 4 * ((k + p) & 7));
}

// 32 consecutive codes (the lower nibble of a byte first) times 32 values vv (float4 k holding
// values 4k .. 4k + 3, in order): sum_i q_i v_i, in eight fp32 partial sums (four packed pairs, one per group of
// 8 inputs: independent chains) that are added at the end.  Packed fp32 pairs: prmt builds the
// float 2^23 + q of a code byte, one packed add takes 2^23 off (exact), one packed fma
// accumulates two products.
__device__ __forceinline__ float q4_dot32(uint4 c, const float4 (&vv)[8]) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
  unsigned long long acc[4] = {0ull, 0ull, 0ull, 0ull};  // fp32 zero pairs
  const unsigned long long neg_magic = 0xCB000000CB000000ull;  // (-2^23, -2^23)
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t t0 = w[k] & 0x0F0F0F0Fu;         // codes of inputs 8k, 8k+2, 8k+4, 8k+6
    const uint32_t t1 = (w[k] >> 4) & 0x0F0F0F0Fu;  // codes of inputs 8k+1, 8k+3, ...
    const float4 a = vv[2 * k];
    const float4 b = vv[2 * k + 1];
    const float xv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const uint32_t sel = (uint32_t)m | (4u << 4) | (5u << 8) | (7u << 12);
      uint32_t lo, hi;
      asm("prmt.b32 %0, %1, %2, %3;" : "=r"(lo) : "r"(t0), "r"(0x4B000000u), "r"(sel));
      asm("prmt.b32 %0, %1, %2, %3;" : "=r"(hi) : "r"(t1), "r"(0x4B000000u), "r"(sel));
      asm("{\n\t.reg .b64 q, x;\n\t"
          "mov.b64 q, {%1, %2};\n\t"
          "mov.b64 x, {%3, %4};\n\t"
          "add.rn.f32x2 q, q, %5;\n\t"
          "fma.rn.f32x2 %0, q, x, %0;\n\t}"
          : "+l"(acc[k])
          : "r"(lo), "r"(hi), "f"(xv[2 * m]), "f"(xv[2 * m + 1]), "l"(neg_magic));
    }
  }
  float sum = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k)
    sum += __uint_as_float((uint32_t)acc[k]) + __uint_as_float((uint32_t)(acc[k] >> 32));
  return sum;
}

// The same with piece p of the swizzled vector v read from shared memory.
__device__ __forceinline__ float q4_dot32(uint4 c, const float* v, int p) {
  float4 vv[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) vv[k] = piece_f4(v, p, k);
  return q4_dot32(c, vv);
}

__device__ __forceinline__ float ld_bf16(const __nv_bfloat16* p) {
  unsigned short u;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(u) : "l"(p));
  return __uint_as_float((uint32_t)u << 16);
}

}  // namespace moe
