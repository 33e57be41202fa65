// CPU oracle of the Gated DeltaNet recurrent scan.  TEST INFRASTRUCTURE ONLY (gdn_oracle.h
// gives the source and the update rule it follows).  fp64, plain loops, one head per task.
#include "gdn_oracle.h"

#include <algorithm>
#include <cstring>
#include <thread>
#include <vector>

namespace {

double widen_bf16(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return (double)f;
}

// One head over all T tokens; S is this head's dk x dv state, updated in place.
void scan_head(const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* alpha,
               const float* beta, int64_t T, int H, int h, int dk, int dv, double* S, double* o) {
  std::vector<double> kt(dk), qt(dk), vt(dv), r(dv), u(dv);
  for (int64_t t = 0; t < T; ++t) {
    const int64_t row = t * H + h;
    for (int i = 0; i < dk; ++i) {
      kt[i] = widen_bf16(k[row * dk + i]);
      qt[i] = widen_bf16(q[row * dk + i]);
    }
    for (int j = 0; j < dv; ++j) vt[j] = widen_bf16(v[row * dv + j]);
    const double a = (double)alpha[row], b = (double)beta[row];
    // decay
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j) S[(int64_t)i * dv + j] *= a;
    // retrieve: r = S^T k
    for (int j = 0; j < dv; ++j) {
      double acc = 0.0;
      for (int i = 0; i < dk; ++i) acc += S[(int64_t)i * dv + j] * kt[i];
      r[j] = acc;
    }
    // delta
    for (int j = 0; j < dv; ++j) u[j] = b * (vt[j] - r[j]);
    // write: S += k u^T
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j) S[(int64_t)i * dv + j] += kt[i] * u[j];
    // read: o = S^T q
    for (int j = 0; j < dv; ++j) {
      double acc = 0.0;
      for (int i = 0; i < dk; ++i) acc += S[(int64_t)i * dv + j] * qt[i];
      o[row * dv + j] = acc;
    }
  }
}

}  // namespace

extern "C" int oracle_gdn_scan(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                               const float* alpha, const float* beta, const float* s0, int64_t T,
                               int H, int dk, int dv, double* o, double* s_out, int nthreads) {
  if (T < 0 || H < 1 || dk < 1 || dv < 1 || !s_out) return -1;
  if (T > 0 && (!q || !k || !v || !alpha || !beta || !o)) return -1;
  const int64_t per = (int64_t)dk * dv;
  for (int64_t e = 0; e < (int64_t)H * per; ++e) s_out[e] = s0 ? (double)s0[e] : 0.0;
  auto run = [&](int h) { scan_head(q, k, v, alpha, beta, T, H, h, dk, dv, s_out + h * per, o); };
  const int nt = std::max(1, std::min(nthreads, H));
  if (nt == 1) {
    for (int h = 0; h < H; ++h) run(h);
    return 0;
  }
  std::vector<std::thread> pool;
  for (int w = 0; w < nt; ++w)
    pool.emplace_back([&, w]() {
      for (int h = w; h < H; h += nt) run(h);
    });
  for (auto& th : pool) th.join();
  return 0;
}
