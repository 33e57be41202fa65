// CPU oracle of the mixture-of-experts FFN layer.  TEST INFRASTRUCTURE ONLY (see
// moe_oracle.h for the sources and the readings it follows).  Plain loops, fp32 arithmetic
// over exactly widened bf16 inputs, fixed summation orders; compiled without fast-math and
// without FMA contraction so that it gives the same bits on every host.
#include "moe_oracle.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <thread>
#include <utility>
#include <vector>

namespace {

float widen(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// fp32 -> bf16, round to nearest, ties to even (finite inputs).
uint16_t round_bf16(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

// Runs fn(i) for i in [0, n) on up to nthreads threads, each index on exactly one thread.
template <class F>
void parallel_for(int64_t n, int nthreads, F fn) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads == 1 || n < 2) {
    for (int64_t i = 0; i < n; ++i) fn(i);
    return;
  }
  int64_t nt = std::min<int64_t>(nthreads, n);
  std::vector<std::thread> pool;
  for (int64_t w = 0; w < nt; ++w) {
    pool.emplace_back([=, &fn]() {
      for (int64_t i = w; i < n; i += nt) fn(i);
    });
  }
  for (auto& t : pool) t.join();
}

// The silu of the gate times the up projection: silu(g) = g / (1 + e^-g).
float swiglu(float g, float u) { return (g / (1.0f + std::exp(-g))) * u; }

// Selection and weights for one row of logits: the k pairs with the largest logit (ties: lower
// id), listed by ascending id; weights exp(l - m) / sum exp(l - m), m = largest kept logit.
void select_row(const float* l, int E, int k, int32_t* idx, float* w) {
  std::vector<std::pair<float, int>> order(E);
  for (int e = 0; e < E; ++e) order[e] = {-l[e], e};
  std::sort(order.begin(), order.end());  // by -logit, then by id
  std::vector<int> kept(k);
  for (int j = 0; j < k; ++j) kept[j] = order[j].second;
  std::sort(kept.begin(), kept.end());
  float m = l[kept[0]];
  for (int j = 1; j < k; ++j) m = std::max(m, l[kept[j]]);
  std::vector<float> ex(k);
  float s = 0.0f;
  for (int j = 0; j < k; ++j) {
    ex[j] = std::exp(l[kept[j]] - m);
    s += ex[j];
  }
  for (int j = 0; j < k; ++j) {
    idx[j] = kept[j];
    w[j] = ex[j] / s;
  }
}

void logits_row_f32(const uint16_t* xr, int d, const uint16_t* w_r, int E, const float* bias,
                    float* out) {
  for (int e = 0; e < E; ++e) {
    const uint16_t* wr = w_r + (int64_t)e * d;
    float acc = 0.0f;
    for (int i = 0; i < d; ++i) acc += widen(xr[i]) * widen(wr[i]);
    out[e] = acc + (bias ? bias[e] : 0.0f);
  }
}

// Weight (r, i) of a bf16 matrix with rows of K elements: the bf16 value widened exactly.
struct Bf16Mat {
  const uint16_t* p;
  int K;
  float operator()(int64_t r, int i) const { return widen(p[r * K + i]); }
};

// Weight (r, i) of a 4-bit group-affine matrix with rows of K elements: code q = nibble i of
// the row (two per byte, the lower nibble first), group g = i / 64; weight = scale_g * q +
// bias_g, one fp32 multiply and one fp32 add.
struct Q4Mat {
  oracle_q4 m;
  int K;
  float operator()(int64_t r, int i) const {
    const uint8_t b = m.codes[r * (K / 2) + i / 2];
    const int q = (i & 1) ? (b >> 4) : (b & 15);
    const int64_t g = r * (K / 64) + i / 64;
    return widen(m.scales[g]) * (float)q + widen(m.biases[g]);
  }
};

// One SwiGLU expert on one row: h[c] = silu(gate_c . x) * (up_c . x) over the d inputs in
// ascending order, then o[n] = down_n . h over the f features in ascending order.
template <class W>
void expert_row_t(const uint16_t* xr, int d, const W& wg, const W& wu, const W& wd, int f,
                  float* h, float* o) {
  for (int c = 0; c < f; ++c) {
    float g = 0.0f, u = 0.0f;
    for (int i = 0; i < d; ++i) g += widen(xr[i]) * wg(c, i);
    for (int i = 0; i < d; ++i) u += widen(xr[i]) * wu(c, i);
    h[c] = swiglu(g, u);
  }
  for (int n = 0; n < d; ++n) {
    float acc = 0.0f;
    for (int c = 0; c < f; ++c) acc += h[c] * wd(n, c);
    o[n] = acc;
  }
}

void expert_row(const uint16_t* xr, int d, const uint16_t* wg, const uint16_t* wu,
                const uint16_t* wd, int f, float* h, float* o) {
  expert_row_t(xr, d, Bf16Mat{wg, d}, Bf16Mat{wu, d}, Bf16Mat{wd, f}, f, h, o);
}

// The layer's output rows for the listed tokens; expert(e, &g, &u, &dn) gives expert e's
// weights (false: not supplied); shared() the shared expert's.
template <class GetExpert, class W>
int forward_t(const oracle_dims* D, const uint16_t* x, int64_t T, const uint16_t* w_r,
              const float* bias, GetExpert expert, const W& sg, const W& su, const W& sd,
              const int64_t* tokens, int64_t n_tokens, uint16_t* y, int32_t* topk_idx,
              float* topk_w, int nthreads) {
  const int d = D->d, E = D->E, k = D->k, f = D->f, fs = D->fs;
  if (!tokens) n_tokens = T;
  for (int64_t r = 0; r < n_tokens; ++r) {
    int64_t t = tokens ? tokens[r] : r;
    if (t < 0 || t >= T) return -1;
  }
  std::vector<int> bad(n_tokens, 0);
  parallel_for(n_tokens, nthreads, [&](int64_t r) {
    int64_t t = tokens ? tokens[r] : r;
    const uint16_t* xr = x + t * d;
    std::vector<float> logits(E), w(k), h(std::max(f, fs)), o(d), acc(d, 0.0f);
    std::vector<int32_t> idx(k);
    logits_row_f32(xr, d, w_r, E, bias, logits.data());
    select_row(logits.data(), E, k, idx.data(), w.data());
    for (int j = 0; j < k; ++j) {  // routed experts in ascending id, weighted
      W g, u, dn;
      if (!expert(idx[j], &g, &u, &dn)) {
        bad[r] = 1;
        return;
      }
      expert_row_t(xr, d, g, u, dn, f, h.data(), o.data());
      for (int n = 0; n < d; ++n) acc[n] += w[j] * o[n];
    }
    expert_row_t(xr, d, sg, su, sd, fs, h.data(), o.data());  // shared, weight 1
    for (int n = 0; n < d; ++n) acc[n] += o[n];
    for (int n = 0; n < d; ++n) y[r * d + n] = round_bf16(acc[n]);
    if (topk_idx)
      for (int j = 0; j < k; ++j) topk_idx[r * k + j] = idx[j];
    if (topk_w)
      for (int j = 0; j < k; ++j) topk_w[r * k + j] = w[j];
  });
  for (int64_t r = 0; r < n_tokens; ++r)
    if (bad[r]) return -3;  // a selected expert's weights were not supplied
  return 0;
}

}  // namespace

extern "C" {

int oracle_router_logits_f64(const uint16_t* x, int64_t T, int d, const uint16_t* w_r, int E,
                             const float* bias, double* logits, int nthreads) {
  if (T < 0 || d <= 0 || E <= 0 || (T > 0 && (!x || !w_r || !logits))) return -1;
  parallel_for(T, nthreads, [&](int64_t t) {
    const uint16_t* xr = x + t * d;
    for (int e = 0; e < E; ++e) {
      const uint16_t* wr = w_r + (int64_t)e * d;
      double acc = 0.0;
      for (int i = 0; i < d; ++i) acc += (double)widen(xr[i]) * (double)widen(wr[i]);
      logits[t * E + e] = acc + (bias ? (double)bias[e] : 0.0);
    }
  });
  return 0;
}

int oracle_router_logits_f32(const uint16_t* x, int64_t T, int d, const uint16_t* w_r, int E,
                             const float* bias, float* logits, int nthreads) {
  if (T < 0 || d <= 0 || E <= 0 || (T > 0 && (!x || !w_r || !logits))) return -1;
  parallel_for(T, nthreads,
               [&](int64_t t) { logits_row_f32(x + t * d, d, w_r, E, bias, logits + t * E); });
  return 0;
}

int oracle_select(const float* logits, int64_t T, int E, int k, int32_t* topk_idx,
                  float* topk_w) {
  if (T < 0 || E <= 0 || k <= 0 || k > E || (T > 0 && (!logits || !topk_idx || !topk_w)))
    return -1;
  for (int64_t t = 0; t < T; ++t) select_row(logits + t * E, E, k, topk_idx + t * k, topk_w + t * k);
  return 0;
}

int oracle_route_structure(const int32_t* topk_idx, int64_t T, int E, int k, int32_t* counts,
                           int32_t* offsets, int32_t* perm, int32_t* inv_perm) {
  if (T < 0 || E <= 0 || k <= 0 || !counts || !offsets) return -1;
  if (T > 0 && (!topk_idx || !perm || !inv_perm)) return -1;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t a = 0; a < T * k; ++a) {
    int e = topk_idx[a];
    if (e < 0 || e >= E) return -2;
    counts[e] += 1;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  // place rows in their expert groups: experts ascending, tokens ascending within a group
  int64_t slot = 0;
  for (int e = 0; e < E; ++e)
    for (int64_t t = 0; t < T; ++t)
      for (int j = 0; j < k; ++j)
        if (topk_idx[t * k + j] == e) {
          perm[slot] = (int32_t)(t * k + j);
          inv_perm[t * k + j] = (int32_t)slot;
          ++slot;
        }
  return 0;
}

int oracle_expert_ffn(const uint16_t* x_row, int d, const uint16_t* w_gate, const uint16_t* w_up,
                      const uint16_t* w_down, int f, float* h, float* o) {
  if (!x_row || !w_gate || !w_up || !w_down || !h || !o || d <= 0 || f <= 0) return -1;
  expert_row(x_row, d, w_gate, w_up, w_down, f, h, o);
  return 0;
}

int oracle_forward(const oracle_dims* D, const uint16_t* x, int64_t T, const uint16_t* w_r,
                   const float* bias, const uint16_t* const* w_gate, const uint16_t* const* w_up,
                   const uint16_t* const* w_down, const uint16_t* ws_gate, const uint16_t* ws_up,
                   const uint16_t* ws_down, const int64_t* tokens, int64_t n_tokens, uint16_t* y,
                   int32_t* topk_idx, float* topk_w, int nthreads) {
  if (!D || D->d <= 0 || D->E <= 0 || D->k <= 0 || D->k > D->E || D->f <= 0 || D->fs <= 0)
    return -1;
  if (T < 0 || !x || !w_r || !w_gate || !w_up || !w_down || !ws_gate || !ws_up || !ws_down || !y)
    return -1;
  const int d = D->d, f = D->f, fs = D->fs;
  auto expert = [&](int e, Bf16Mat* g, Bf16Mat* u, Bf16Mat* dn) {
    if (!w_gate[e] || !w_up[e] || !w_down[e]) return false;
    *g = Bf16Mat{w_gate[e], d};
    *u = Bf16Mat{w_up[e], d};
    *dn = Bf16Mat{w_down[e], f};
    return true;
  };
  return forward_t(D, x, T, w_r, bias, expert, Bf16Mat{ws_gate, d}, Bf16Mat{ws_up, d},
                   Bf16Mat{ws_down, fs}, tokens, n_tokens, y, topk_idx, topk_w, nthreads);
}

int oracle_dequant_q4(const oracle_q4* m, int64_t rows, int K, float* out) {
  if (!m || !m->codes || !m->scales || !m->biases || !out || rows < 0 || K <= 0 || K % 64)
    return -1;
  const Q4Mat w{*m, K};
  for (int64_t r = 0; r < rows; ++r)
    for (int i = 0; i < K; ++i) out[r * K + i] = w(r, i);
  return 0;
}

int oracle_forward_q4(const oracle_dims* D, const uint16_t* x, int64_t T, const uint16_t* w_r,
                      const float* bias, const oracle_q4* w_gate, const oracle_q4* w_up,
                      const oracle_q4* w_down, const oracle_q4* ws_gate, const oracle_q4* ws_up,
                      const oracle_q4* ws_down, const int64_t* tokens, int64_t n_tokens,
                      uint16_t* y, int32_t* topk_idx, float* topk_w, int nthreads) {
  if (!D || D->d <= 0 || D->E <= 0 || D->k <= 0 || D->k > D->E || D->f <= 0 || D->fs <= 0)
    return -1;
  if (D->d % 64 || D->f % 64 || D->fs % 64) return -1;
  if (T < 0 || !x || !w_r || !w_gate || !w_up || !w_down || !ws_gate || !ws_up || !ws_down || !y)
    return -1;
  if (!ws_gate->codes || !ws_up->codes || !ws_down->codes) return -1;
  const int d = D->d, f = D->f, fs = D->fs;
  auto expert = [&](int e, Q4Mat* g, Q4Mat* u, Q4Mat* dn) {
    if (!w_gate[e].codes || !w_up[e].codes || !w_down[e].codes) return false;
    *g = Q4Mat{w_gate[e], d};
    *u = Q4Mat{w_up[e], d};
    *dn = Q4Mat{w_down[e], f};
    return true;
  };
  return forward_t(D, x, T, w_r, bias, expert, Q4Mat{*ws_gate, d}, Q4Mat{*ws_up, d},
                   Q4Mat{*ws_down, fs}, tokens, n_tokens, y, topk_idx, topk_w, nthreads);
}

}  // extern "C"
