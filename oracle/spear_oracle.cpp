// spear_oracle.cpp -- plain CPU reference for the gated W4 + low-rank
// error-compensated linear layer ("SPEAR", gist.science explainer, Technical
// Summary 2.1 A "Input-Adaptive Error Compensators" and 2.1 B "CKA-Guided
// Entropy-Aware Module Selection").
//
// TEST INFRASTRUCTURE ONLY: the parity oracle.  It is independent of the CUDA
// library (no shared code, headers or tables) and is loaded only by the tests,
// the smoke check and the benchmark's CPU-baseline leg.
//
// Every function is a direct, literal statement of the definition: one loop
// per sum, no blocking or reordering.  Build with -ffp-contract=off so that
// float expressions are evaluated exactly as written.

#include "spear_oracle.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <functional>
#include <thread>
#include <vector>

namespace {

uint32_t float_bits(float f) { uint32_t u; std::memcpy(&u, &f, 4); return u; }
float bits_float(uint32_t u) { float f; std::memcpy(&f, &u, 4); return f; }

// ---------------------------------------------------------------- numbers --

// IEEE binary16 from a float, rounding toward +infinity.  The scale of every
// quantisation group is stored this way so that it is never smaller than the
// exact fp32 quotient (which keeps every code inside its range).
uint16_t f32_to_f16_ru(float f) {
  uint32_t b = float_bits(f);
  uint32_t sign = b >> 31;
  uint32_t e8 = (b >> 23) & 0xFF;
  uint32_t m23 = b & 0x7FFFFF;
  if (e8 == 0xFF) {                         // inf or nan
    if (m23) return 0x7E00;
    return sign ? 0xFC00 : 0x7C00;
  }
  if (e8 == 0) {                            // float zero or float subnormal
    if (m23 == 0) return (uint16_t)(sign << 15);
    return sign ? 0x8000 : 0x0001;          // tiny: -0 (toward +inf) or min subnormal
  }
  int e = (int)e8 - 127;
  uint32_t h;
  bool inexact;
  if (e > 15) {                             // beyond the binary16 range
    return sign ? 0xFBFF : 0x7C00;          // -65504 or +inf
  } else if (e >= -14) {                    // binary16 normal
    h = ((uint32_t)(e + 15) << 10) | (m23 >> 13);
    inexact = (m23 & 0x1FFF) != 0;
  } else {                                  // binary16 subnormal, unit 2^-24
    uint32_t m24 = (1u << 23) | m23;        // value = m24 * 2^(e-23)
    int s = -e - 1;                         // value / 2^-24 = m24 >> s
    if (s >= 32) { h = 0; inexact = true; }
    else { h = m24 >> s; inexact = (m24 & ((1u << s) - 1)) != 0; }
  }
  if (inexact && !sign) h += 1;             // toward +inf: bump magnitude of positives
  return (uint16_t)((sign << 15) | h);
}

float f16_to_f32(uint16_t h) {
  uint32_t sign = (uint32_t)(h >> 15) << 31;
  uint32_t e5 = (h >> 10) & 0x1F;
  uint32_t m10 = h & 0x3FF;
  if (e5 == 0x1F) return bits_float(sign | 0x7F800000u | (m10 << 13));
  if (e5 == 0) {                            // zero or subnormal: m10 * 2^-24
    float v = (float)m10 * std::ldexp(1.0f, -24);
    return sign ? -v : v;
  }
  return bits_float(sign | ((e5 - 15 + 127) << 23) | (m10 << 13));
}

uint16_t f32_to_bf16_rn(float f) {
  uint32_t b = float_bits(f);
  if ((b & 0x7F800000u) == 0x7F800000u && (b & 0x7FFFFF)) return 0x7FC0;
  uint32_t lsb = (b >> 16) & 1;
  b += 0x7FFF + lsb;                        // round half to even
  return (uint16_t)(b >> 16);
}

float bf16_to_f32(uint16_t v) { return bits_float((uint32_t)v << 16); }

// ------------------------------------------------------------ quantiser ---

int nibble(const uint8_t* row, int i) {
  uint8_t byte = row[i >> 1];
  return (i & 1) ? (byte >> 4) : (byte & 0xF);
}

void set_nibble(uint8_t* row, int i, int v) {
  uint8_t& byte = row[i >> 1];
  if (i & 1) byte = (uint8_t)((byte & 0x0F) | (v << 4));
  else       byte = (uint8_t)((byte & 0xF0) | v);
}

int round_half_even(float v) { return (int)std::nearbyint(v); }

int clampi(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }

bool shape_ok(int N, int K, int G) {
  return N > 0 && K > 0 && G > 0 && K % G == 0 && K % 2 == 0;
}

// Splits [0, count) into contiguous slices, one std::thread each.
void parallel_rows(int count, int nthreads, const std::function<void(int, int)>& body) {
  if (nthreads <= 1 || count < 2) { body(0, count); return; }
  int t = std::min(nthreads, count);
  std::vector<std::thread> pool;
  for (int i = 0; i < t; ++i) {
    int a = (int)((long long)count * i / t), b = (int)((long long)count * (i + 1) / t);
    pool.emplace_back(body, a, b);
  }
  for (auto& th : pool) th.join();
}
}  // namespace

extern "C" {

uint16_t oracle_f32_to_f16_ru(float f) { return f32_to_f16_ru(f); }
float oracle_f16_to_f32(uint16_t h) { return f16_to_f32(h); }
uint16_t oracle_f32_to_bf16_rn(float f) { return f32_to_bf16_rn(f); }
float oracle_bf16_to_f32(uint16_t b) { return bf16_to_f32(b); }

int oracle_quantize_pack(const float* W, int N, int K, int G, int sym,
                         uint8_t* qweight, uint16_t* scales, uint8_t* zeros) {
  if (!W || !qweight || !scales || !shape_ok(N, K, G)) return 1;
  if (!sym && !zeros) return 1;
  const int ng = K / G;
  const int zrow = (ng + 1) / 2;
  std::memset(qweight, 0, (size_t)N * (K / 2));
  if (!sym) std::memset(zeros, 0, (size_t)N * zrow);
  for (int n = 0; n < N; ++n) {
    const float* w = W + (size_t)n * K;
    uint8_t* qrow = qweight + (size_t)n * (K / 2);
    for (int gi = 0; gi < ng; ++gi) {
      const int k0 = gi * G;
      for (int k = k0; k < k0 + G; ++k)
        if (!std::isfinite(w[k])) return 1;
      if (sym) {
        // scale: the largest magnitude maps onto code +-7
        float amax = 0.0f;
        for (int k = k0; k < k0 + G; ++k) amax = std::max(amax, std::fabs(w[k]));
        float s32 = amax / 7.0f;
        uint16_t s16 = f32_to_f16_ru(s32);
        if (s16 == 0x7C00) return 1;                      // scale overflows fp16
        float s = f16_to_f32(s16);
        scales[(size_t)n * ng + gi] = s16;
        for (int k = k0; k < k0 + G; ++k) {
          int u = 8;                                      // all-zero group
          if (s != 0.0f) u = clampi(round_half_even(w[k] / s), -8, 7) + 8;
          set_nibble(qrow, k, u);
        }
      } else {
        // range [lo, hi] always contains 0, so 0 is on the grid
        float lo = 0.0f, hi = 0.0f;
        for (int k = k0; k < k0 + G; ++k) { lo = std::min(lo, w[k]); hi = std::max(hi, w[k]); }
        float s32 = (hi - lo) / 15.0f;
        uint16_t s16 = f32_to_f16_ru(s32);
        if (s16 == 0x7C00) return 1;
        float s = f16_to_f32(s16);
        scales[(size_t)n * ng + gi] = s16;
        int z = 0;
        if (s != 0.0f) z = clampi(round_half_even(-lo / s), 0, 15);
        set_nibble(zeros + (size_t)n * zrow, gi, z);
        for (int k = k0; k < k0 + G; ++k) {
          int u = 0;
          if (s != 0.0f) u = clampi(round_half_even(w[k] / s) + z, 0, 15);
          set_nibble(qrow, k, u);
        }
      }
    }
  }
  return 0;
}

int oracle_unpack_codes(const uint8_t* qweight, int N, int K, uint8_t* codes) {
  if (!qweight || !codes || N <= 0 || K <= 0 || K % 2) return 1;
  for (int n = 0; n < N; ++n)
    for (int k = 0; k < K; ++k)
      codes[(size_t)n * K + k] = (uint8_t)nibble(qweight + (size_t)n * (K / 2), k);
  return 0;
}

int oracle_unpack_zeros(const uint8_t* zeros, int N, int K, int G, int sym, uint8_t* z) {
  if (!z || !shape_ok(N, K, G) || (!sym && !zeros)) return 1;
  const int ng = K / G, zrow = (ng + 1) / 2;
  for (int n = 0; n < N; ++n)
    for (int gi = 0; gi < ng; ++gi)
      z[(size_t)n * ng + gi] = sym ? 8 : (uint8_t)nibble(zeros + (size_t)n * zrow, gi);
  return 0;
}

int oracle_dequant(const uint8_t* qweight, const uint16_t* scales, const uint8_t* zeros,
                   int N, int K, int G, int sym, double* dq) {
  if (!qweight || !scales || !dq || !shape_ok(N, K, G) || (!sym && !zeros)) return 1;
  const int ng = K / G, zrow = (ng + 1) / 2;
  for (int n = 0; n < N; ++n)
    for (int k = 0; k < K; ++k) {
      int gi = k / G;
      int u = nibble(qweight + (size_t)n * (K / 2), k);
      int z = sym ? 8 : nibble(zeros + (size_t)n * zrow, gi);
      double s = (double)f16_to_f32(scales[(size_t)n * ng + gi]);
      dq[(size_t)n * K + k] = (double)(u - z) * s;
    }
  return 0;
}

int oracle_linear(int N, int K, int G, int sym,
                  const uint8_t* qweight, const uint16_t* scales, const uint8_t* zeros,
                  int r, const uint16_t* A, const uint16_t* B, const uint16_t* w_g,
                  float b_g, float alpha, int comp_enabled,
                  const uint16_t* x, int M,
                  const int* n_idx, int n_count,
                  int accum_double, int nthreads,
                  double* y, double* corr, double* gate) {
  if (!qweight || !scales || !x || !y || !shape_ok(N, K, G) || M < 0 || r < 0) return 1;
  if (!sym && !zeros) return 1;
  const bool comp = comp_enabled && r > 0;
  if (comp && (!A || !B || !w_g)) return 1;
  const int cols = n_idx ? n_count : N;
  if (cols < 0) return 1;
  if (n_idx)
    for (int i = 0; i < cols; ++i)
      if (n_idx[i] < 0 || n_idx[i] >= N) return 1;
  const int ng = K / G, zrow = (ng + 1) / 2;

  // Per-token gate g_m and down-projection t_m = A x_m.
  std::vector<double> g(M, 0.0), t((size_t)M * (r > 0 ? r : 1), 0.0);
  for (int m = 0; m < M; ++m) {
    const uint16_t* xm = x + (size_t)m * K;
    if (!comp) continue;
    double s;
    if (accum_double) {
      s = 0.0;
      for (int k = 0; k < K; ++k) s += (double)bf16_to_f32(w_g[k]) * (double)bf16_to_f32(xm[k]);
      s += (double)b_g;
    } else {
      float sf = 0.0f;
      for (int k = 0; k < K; ++k) sf = sf + bf16_to_f32(w_g[k]) * bf16_to_f32(xm[k]);
      s = (double)(sf + b_g);
    }
    g[m] = 1.0 / (1.0 + std::exp(-s));
    for (int j = 0; j < r; ++j) {
      const uint16_t* aj = A + (size_t)j * K;
      if (accum_double) {
        double acc = 0.0;
        for (int k = 0; k < K; ++k) acc += (double)bf16_to_f32(aj[k]) * (double)bf16_to_f32(xm[k]);
        t[(size_t)m * r + j] = acc;
      } else {
        float acc = 0.0f;
        for (int k = 0; k < K; ++k) acc = acc + bf16_to_f32(aj[k]) * bf16_to_f32(xm[k]);
        t[(size_t)m * r + j] = (double)acc;
      }
    }
  }
  if (gate) for (int m = 0; m < M; ++m) gate[m] = comp ? g[m] : 0.0;

  auto body = [&](int c0, int c1) {
    std::vector<double> dq(K);
    for (int c = c0; c < c1; ++c) {
      const int n = n_idx ? n_idx[c] : c;
      const uint8_t* qrow = qweight + (size_t)n * (K / 2);
      for (int k = 0; k < K; ++k) {
        int gi = k / G;
        int u = nibble(qrow, k);
        int z = sym ? 8 : nibble(zeros + (size_t)n * zrow, gi);
        dq[k] = (double)(u - z) * (double)f16_to_f32(scales[(size_t)n * ng + gi]);
      }
      for (int m = 0; m < M; ++m) {
        const uint16_t* xm = x + (size_t)m * K;
        double main_term;
        if (accum_double) {
          double acc = 0.0;
          for (int k = 0; k < K; ++k) acc += dq[k] * (double)bf16_to_f32(xm[k]);
          main_term = acc;
        } else {
          float acc = 0.0f;
          for (int k = 0; k < K; ++k) acc = acc + (float)dq[k] * bf16_to_f32(xm[k]);
          main_term = (double)acc;
        }
        double c_term = 0.0;
        if (comp) {
          double bt = 0.0;
          for (int j = 0; j < r; ++j)
            bt += (double)bf16_to_f32(B[(size_t)n * r + j]) * t[(size_t)m * r + j];
          c_term = (double)alpha * g[m] * bt;
        }
        y[(size_t)m * cols + c] = main_term + c_term;
        if (corr) corr[(size_t)m * cols + c] = c_term;
      }
    }
  };
  parallel_rows(cols, nthreads, body);
  return 0;
}

int oracle_linear_vector_gate(int N, int K, int G, int sym,
                              const uint8_t* qweight, const uint16_t* scales, const uint8_t* zeros,
                              int r, const uint16_t* A, const uint16_t* B,
                              int h, const float* W1, const float* c1,
                              const float* W2, const float* c2, float alpha,
                              const uint16_t* x, int M, int nthreads,
                              double* y, double* gamma_out) {
  if (!qweight || !scales || !x || !y || !A || !B || !W1 || !c1 || !W2 || !c2) return 1;
  if (!shape_ok(N, K, G) || M < 0 || r <= 0 || h <= 0 || (!sym && !zeros)) return 1;
  const int ng = K / G, zrow = (ng + 1) / 2;
  // u_m = diag(gamma(t_m)) t_m with t_m = A x_m, gamma = sigmoid(W2 relu(W1 t + c1) + c2)
  std::vector<double> u((size_t)M * r);
  for (int m = 0; m < M; ++m) {
    const uint16_t* xm = x + (size_t)m * K;
    std::vector<double> t(r), hid(h);
    for (int j = 0; j < r; ++j) {
      double acc = 0.0;
      for (int k = 0; k < K; ++k) acc += (double)bf16_to_f32(A[(size_t)j * K + k]) * (double)bf16_to_f32(xm[k]);
      t[j] = acc;
    }
    for (int i = 0; i < h; ++i) {
      double acc = (double)c1[i];
      for (int j = 0; j < r; ++j) acc += (double)W1[(size_t)i * r + j] * t[j];
      hid[i] = acc > 0.0 ? acc : 0.0;
    }
    for (int j = 0; j < r; ++j) {
      double acc = (double)c2[j];
      for (int i = 0; i < h; ++i) acc += (double)W2[(size_t)j * h + i] * hid[i];
      double gj = 1.0 / (1.0 + std::exp(-acc));
      if (gamma_out) gamma_out[(size_t)m * r + j] = gj;
      u[(size_t)m * r + j] = gj * t[j];
    }
  }
  auto body = [&](int n0, int n1) {
    std::vector<double> dq(K);
    for (int n = n0; n < n1; ++n) {
      for (int k = 0; k < K; ++k) {
        int gi = k / G;
        int uq = nibble(qweight + (size_t)n * (K / 2), k);
        int z = sym ? 8 : nibble(zeros + (size_t)n * zrow, gi);
        dq[k] = (double)(uq - z) * (double)f16_to_f32(scales[(size_t)n * ng + gi]);
      }
      for (int m = 0; m < M; ++m) {
        double acc = 0.0;
        for (int k = 0; k < K; ++k) acc += dq[k] * (double)bf16_to_f32(x[(size_t)m * K + k]);
        double bu = 0.0;
        for (int j = 0; j < r; ++j) bu += (double)bf16_to_f32(B[(size_t)n * r + j]) * u[(size_t)m * r + j];
        y[(size_t)m * N + n] = acc + (double)alpha * bu;
      }
    }
  };
  parallel_rows(N, nthreads, body);
  return 0;
}

int oracle_layer_select_mask(const float* damage, const float* cost, int L,
                             double budget_bytes, int rank_min, int rank_max,
                             uint8_t* mask_out, int* rank_out) {
  if (!damage || !cost || !mask_out || !rank_out || L <= 0) return 1;
  if (rank_min <= 0 || rank_max < rank_min || !(budget_bytes >= 0.0)) return 1;
  for (int i = 0; i < L; ++i) {
    if (!std::isfinite(damage[i]) || damage[i] < 0.0f) return 1;
    if (!std::isfinite(cost[i]) || cost[i] <= 0.0f) return 1;
  }
  for (int i = 0; i < L; ++i) { mask_out[i] = 0; rank_out[i] = 0; }

  double dsum = 0.0, csum = 0.0;
  for (int i = 0; i < L; ++i) { dsum += damage[i]; csum += cost[i]; }
  if (dsum <= 0.0) return 0;                      // nothing is damaged
  const double cmean = csum / L;

  // damage distribution and its entropy
  std::vector<double> p(L);
  for (int i = 0; i < L; ++i) p[i] = damage[i] / dsum;
  double H = 0.0;
  for (int i = 0; i < L; ++i) if (p[i] > 0.0) H -= p[i] * std::log(p[i]);
  int k = (int)std::floor(std::exp(H) + 0.5);     // effective number of damaged modules
  k = clampi(k, 1, L);

  // hybrid score: damage share per unit of relative deployment cost
  std::vector<int> order(L);
  for (int i = 0; i < L; ++i) order[i] = i;
  std::vector<double> score(L);
  for (int i = 0; i < L; ++i) score[i] = p[i] / (cost[i] / cmean);
  std::stable_sort(order.begin(), order.end(),
                   [&](int a, int b) { return score[a] > score[b]; });

  // smallest allowed rank: first multiple of 16 at or above rank_min
  const int rlo = ((rank_min + 15) / 16) * 16;
  const int rhi = (rank_max / 16) * 16;
  if (rlo > rhi) return 1;

  for (int take = k; take >= 1; --take) {
    double sel_cost = 0.0;
    for (int i = 0; i < take; ++i) sel_cost += cost[order[i]];
    int best = 0;
    for (int rr = rhi; rr >= rlo; rr -= 16)
      if ((double)rr * sel_cost <= budget_bytes) { best = rr; break; }
    if (best > 0) {
      for (int i = 0; i < take; ++i) { mask_out[order[i]] = 1; rank_out[order[i]] = best; }
      return 0;
    }
  }
  return 0;                                       // budget too small for any module
}

}  // extern "C"
