// cka.cu -- linear centred kernel alignment on the host (SPEAR explainer,
// Technical Summary 2.1 B: CKA as the training-free proxy for the damage that
// quantising a module does; the module-selection rule takes the damage scores).
//
//   X [n][dx], Y [n][dy] (one row per token), columns centred to Xc, Yc:
//   CKA(X, Y) = <Xc Xc^T, Yc Yc^T>_F / (||Xc Xc^T||_F ||Yc Yc^T||_F)
//             = ||Xc^T Yc||_F^2 / (||Xc^T Xc||_F ||Yc^T Yc||_F)
// Both forms are the same number; the token-space one (n x n Grams) is used
// when n is at most the feature width, the feature-space one otherwise.
// fp64 throughout, rows of each product split over the hardware threads.
#include <algorithm>
#include <cmath>
#include <functional>
#include <thread>
#include <vector>

#include "internal.h"

namespace spear {
namespace {

void parallel_rows(int rows, const std::function<void(int, int)>& body) {
  const int nt = std::max(1, std::min<int>((int)std::thread::hardware_concurrency(), rows / 8 + 1));
  if (nt == 1) {
    body(0, rows);
    return;
  }
  std::vector<std::thread> th;
  for (int t = 0; t < nt; ++t) th.emplace_back(body, (int)((long long)rows * t / nt), (int)((long long)rows * (t + 1) / nt));
  for (auto& x : th) x.join();
}

// Column-centred copy of a [n][d] fp32 matrix, fp64.
std::vector<double> centred(const float* A, int n, int d) {
  std::vector<double> out((size_t)n * d), mean(d, 0.0);
  for (int i = 0; i < n; ++i)
    for (int j = 0; j < d; ++j) mean[j] += A[(size_t)i * d + j];
  for (int j = 0; j < d; ++j) mean[j] /= n;
  for (int i = 0; i < n; ++i)
    for (int j = 0; j < d; ++j) out[(size_t)i * d + j] = A[(size_t)i * d + j] - mean[j];
  return out;
}

// G = A^T B for A [n][da], B [n][db] (feature space) or A B^T for A [n][d],
// B [n][d] (token space); returned row-major.
std::vector<double> gram_tokens(const std::vector<double>& A, const std::vector<double>& B, int n, int d) {
  std::vector<double> G((size_t)n * n);
  parallel_rows(n, [&](int i0, int i1) {
    for (int i = i0; i < i1; ++i)
      for (int j = 0; j < n; ++j) {
        double s = 0.0;
        const double* a = &A[(size_t)i * d];
        const double* b = &B[(size_t)j * d];
        for (int k = 0; k < d; ++k) s += a[k] * b[k];
        G[(size_t)i * n + j] = s;
      }
  });
  return G;
}
std::vector<double> gram_features(const std::vector<double>& A, const std::vector<double>& B, int n, int da, int db) {
  std::vector<double> G((size_t)da * db, 0.0);
  parallel_rows(da, [&](int i0, int i1) {
    for (int t = 0; t < n; ++t) {
      const double* a = &A[(size_t)t * da];
      const double* b = &B[(size_t)t * db];
      for (int i = i0; i < i1; ++i) {
        const double ai = a[i];
        double* g = &G[(size_t)i * db];
        for (int j = 0; j < db; ++j) g[j] += ai * b[j];
      }
    }
  });
  return G;
}
double dot(const std::vector<double>& a, const std::vector<double>& b) {
  double s = 0.0;
  for (size_t i = 0; i < a.size(); ++i) s += a[i] * b[i];
  return s;
}

}  // namespace
}  // namespace spear

using namespace spear;

spear_status spear_linear_cka(const float* X, const float* Y, int n, int dx, int dy, double* cka_out) {
  if (!X || !Y || !cka_out || n < 2 || dx < 1 || dy < 1)
    return fail(SPEAR_ERR_INVALID_ARG, "linear_cka: need n >= 2 tokens and non-empty X, Y");
  for (size_t i = 0; i < (size_t)n * dx; ++i)
    if (!std::isfinite(X[i])) return fail(SPEAR_ERR_INVALID_ARG, "linear_cka: X has a non-finite value");
  for (size_t i = 0; i < (size_t)n * dy; ++i)
    if (!std::isfinite(Y[i])) return fail(SPEAR_ERR_INVALID_ARG, "linear_cka: Y has a non-finite value");
  const std::vector<double> Xc = centred(X, n, dx), Yc = centred(Y, n, dy);
  double xy, xx, yy;
  if (n <= std::max(dx, dy)) {
    const std::vector<double> K = gram_tokens(Xc, Xc, n, dx), L = gram_tokens(Yc, Yc, n, dy);
    xy = dot(K, L);
    xx = dot(K, K);
    yy = dot(L, L);
  } else {
    const std::vector<double> Cxy = gram_features(Xc, Yc, n, dx, dy);
    const std::vector<double> Cxx = gram_features(Xc, Xc, n, dx, dx), Cyy = gram_features(Yc, Yc, n, dy, dy);
    xy = dot(Cxy, Cxy);
    xx = dot(Cxx, Cxx);
    yy = dot(Cyy, Cyy);
  }
  if (!(xx > 0.0) || !(yy > 0.0)) return fail(SPEAR_ERR_INVALID_ARG, "linear_cka: X or Y has no variance");
  *cka_out = xy / std::sqrt(xx * yy);
  return SPEAR_OK;
}

spear_status spear_cka_damage(const float* X_ref, const float* Y_quant, int n, int dx, int dy, double* damage_out) {
  if (!damage_out) return fail(SPEAR_ERR_INVALID_ARG, "cka_damage: damage_out is NULL");
  double cka = 0.0;
  if (spear_status rc = spear_linear_cka(X_ref, Y_quant, n, dx, dy, &cka)) return rc;
  *damage_out = 1.0 - cka;
  return SPEAR_OK;
}
