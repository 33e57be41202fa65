/* Host half of the seeded input generator; the definitions are in synth.h. */
#include "synth.h"

#include <pthread.h>
#include <string.h>

#define SM64_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t sm64_fin(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

uint64_t synth_key(uint64_t seed, uint64_t stream) {
  return sm64_fin(sm64_fin(seed) + stream * SM64_GAMMA);
}

uint64_t synth_word(uint64_t key, uint64_t i) { return sm64_fin(key + (i + 1) * SM64_GAMMA); }

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static inline uint16_t normal_element(uint64_t key, uint64_t idx, float sigma) {
  int32_t s = 0;
  for (int w = 0; w < 3; ++w) {
    uint64_t v = synth_word(key, 3 * idx + (uint64_t)w);
    for (int q = 0; q < 4; ++q) s += (int32_t)((v >> (16 * q)) & 0xFFFFu);
  }
  int32_t n = s - 393210;
  float z = (float)n * 0x1p-16f; /* exact: |n| < 2^20 */
  return f32_to_bf16_rne(z * sigma);
}

typedef struct {
  uint64_t key, offset, begin, end;
  float sigma;
  uint16_t* out;
} chunk_t;

static void* run_chunk(void* p) {
  chunk_t* c = (chunk_t*)p;
  for (uint64_t j = c->begin; j < c->end; ++j) c->out[j] = normal_element(c->key, c->offset + j, c->sigma);
  return NULL;
}

void synth_normal_bf16(uint64_t seed, uint64_t stream, uint64_t offset, uint64_t n, float sigma,
                       uint16_t* out, int nthreads) {
  uint64_t key = synth_key(seed, stream);
  if (nthreads <= 1 || n < (1u << 16)) {
    chunk_t c = {key, offset, 0, n, sigma, out};
    run_chunk(&c);
    return;
  }
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  chunk_t cs[256];
  uint64_t per = (n + (uint64_t)nthreads - 1) / (uint64_t)nthreads;
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    uint64_t b = per * (uint64_t)t, e = b + per;
    if (b >= n) break;
    if (e > n) e = n;
    cs[t] = (chunk_t){key, offset, b, e, sigma, out};
    if (pthread_create(&th[t], NULL, run_chunk, &cs[t]) != 0) {
      run_chunk(&cs[t]); /* no thread available: do the chunk here */
      th[t] = 0;
    }
    started = t + 1;
  }
  for (int t = 0; t < started; ++t)
    if (th[t]) pthread_join(th[t], NULL);
}

void synth_permutation(uint64_t seed, uint64_t stream, int32_t n, int32_t* out) {
  uint64_t key = synth_key(seed, stream), ctr = 0;
  for (int32_t i = 0; i < n; ++i) out[i] = i;
  for (int32_t i = n - 1; i > 0; --i) {
    uint64_t m = (uint64_t)i + 1;
    /* accept w only below the largest multiple of m that fits, so w % m is uniform */
    uint64_t bound = (UINT64_MAX / m) * m;
    uint64_t w;
    do { w = synth_word(key, ctr++); } while (w >= bound);
    int32_t j = (int32_t)(w % m);
    int32_t t = out[i];
    out[i] = out[j];
    out[j] = t;
  }
}

void synth_bytes(uint64_t seed, uint64_t stream, uint64_t offset, uint64_t n, uint8_t* out) {
  uint64_t key = synth_key(seed, stream);
  for (uint64_t j = 0; j < n; ++j) {
    uint64_t b = offset + j;
    out[j] = (uint8_t)(synth_word(key, b >> 3) >> (8 * (b & 7)));
  }
}

void synth_q4_affine(uint64_t seed, uint64_t stream, uint64_t offset, uint64_t n, float base,
                     uint16_t* scales, uint16_t* biases) {
  uint64_t key = synth_key(seed, stream);
  for (uint64_t j = 0; j < n; ++j) {
    uint32_t u = (uint32_t)(synth_word(key, offset + j) >> 41);
    float v = 0.75f + (float)u * 0x1p-24f;
    uint16_t sb = f32_to_bf16_rne(v * base);
    scales[j] = sb;
    biases[j] = (uint16_t)(sb ^ 0x8000u) + (uint16_t)(3u << 7); /* -8 s: sign flip, exponent + 3 */
  }
}

void synth_uniform_f32(uint64_t seed, uint64_t stream, uint64_t offset, uint64_t n, float lo,
                       float hi, float* out) {
  uint64_t key = synth_key(seed, stream);
  const float span = hi - lo;
  for (uint64_t j = 0; j < n; ++j) {
    float u = (float)(uint32_t)(synth_word(key, offset + j) >> 40) * 0x1p-24f;
    float p = span * u;
    out[j] = lo + p;
  }
}
