// api.cu -- the library's C ABI (include/spear.h): argument checks, error
// reporting, phase dispatch and the host-side module selection.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <numeric>
#include <vector>

#include "internal.h"

namespace spear {

namespace {
thread_local char t_last_error[512] = "";

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

bool rank_ok(int r) { return r == 0 || r == 16 || r == 32 || r == 64; }

int check_shape(int N, int K, int G) {
  if (N <= 0 || K <= 0) return fail(SPEAR_ERR_INVALID_ARG, "N=%d, K=%d must be positive", N, K);
  if (K % 128) return fail(SPEAR_ERR_INVALID_ARG, "K=%d must be a multiple of 128", K);
  if (N % 64) return fail(SPEAR_ERR_INVALID_ARG, "N=%d must be a multiple of 64", N);
  if (G != K && G != 128) return fail(SPEAR_ERR_INVALID_ARG, "group_size=%d must be K or 128", G);
  return SPEAR_OK;
}

int check_layer(const spear_w4_layer* L) {
  if (!L) return fail(SPEAR_ERR_INVALID_ARG, "layer is NULL");
  if (int rc = check_shape(L->N, L->K, L->group_size)) return rc;
  if (!L->qweight || !L->scales) return fail(SPEAR_ERR_INVALID_ARG, "qweight/scales are NULL");
  if (!L->symmetric && !L->zeros) return fail(SPEAR_ERR_INVALID_ARG, "asymmetric layer needs zeros");
  if (!aligned16(L->qweight) || !aligned16(L->scales) || (L->zeros && !aligned16(L->zeros)))
    return fail(SPEAR_ERR_INVALID_ARG, "layer buffers must be 16-byte aligned");
  if (!rank_ok(L->rank)) return fail(SPEAR_ERR_INVALID_ARG, "rank=%d must be 0, 16, 32 or 64", L->rank);
  if (L->gate_hidden < 0 || L->gate_hidden > 32)
    return fail(SPEAR_ERR_INVALID_ARG, "gate_hidden=%d must be in [0, 32]", L->gate_hidden);
  if (L->comp_enabled && L->rank > 0) {
    const bool vec = L->gate_hidden > 0;
    if (!L->A || !L->B || (!vec && !L->w_g)) return fail(SPEAR_ERR_INVALID_ARG, "compensator buffers are NULL");
    if (!aligned16(L->A) || !aligned16(L->B) || (L->w_g && !aligned16(L->w_g)))
      return fail(SPEAR_ERR_INVALID_ARG, "compensator buffers must be 16-byte aligned");
    if (vec && (!L->gate_w1 || !L->gate_c1 || !L->gate_w2 || !L->gate_c2))
      return fail(SPEAR_ERR_INVALID_ARG, "vector-gate buffers are NULL");
    if (vec && (!aligned16(L->gate_w1) || !aligned16(L->gate_c1) || !aligned16(L->gate_w2) ||
                !aligned16(L->gate_c2)))
      return fail(SPEAR_ERR_INVALID_ARG, "vector-gate buffers must be 16-byte aligned");
    if (!std::isfinite(L->alpha) || (!vec && std::isnan(L->b_g)))
      return fail(SPEAR_ERR_INVALID_ARG, "alpha must be finite and b_g not NaN");
  }
  return SPEAR_OK;
}
}  // namespace

void set_last_error(const char* msg) { snprintf(t_last_error, sizeof(t_last_error), "%s", msg ? msg : ""); }

int fail(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
  va_end(ap);
  return status;
}

int cuda_check(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return SPEAR_OK;
  return fail(SPEAR_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

namespace {
std::atomic<bool> g_launch_overlap{false};
std::atomic<uint64_t> g_wait_limit_ns{0};
}  // namespace

void set_launch_overlap(bool on) { g_launch_overlap.store(on); }
bool launch_overlap() { return g_launch_overlap.load(); }
uint64_t wait_limit_ns(uint64_t default_ns) {
  const uint64_t v = g_wait_limit_ns.load();
  return v ? v : default_ns;
}

bool log_plans() {
  static const bool on = [] {
    const char* v = std::getenv("SPEAR_LOG_PLANS");
    return v && v[0] && std::strcmp(v, "0") != 0;
  }();
  return on;
}

int ensure_smem_limit(const void* fn, size_t bytes) {
  struct Entry { int device; const void* fn; size_t bytes; };
  static std::mutex mu;
  static std::vector<Entry> limits;
  int dev = 0;
  if (int rc = cuda_check(cudaGetDevice(&dev), "cudaGetDevice")) return rc;
  std::lock_guard<std::mutex> lk(mu);
  for (Entry& e : limits)
    if (e.device == dev && e.fn == fn) {
      if (bytes <= e.bytes) return SPEAR_OK;
      if (int rc = cuda_check(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes),
                              "shared-memory limit")) return rc;
      e.bytes = bytes;
      return SPEAR_OK;
    }
  if (int rc = cuda_check(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes),
                          "shared-memory limit")) return rc;
  limits.push_back({dev, fn, bytes});
  return SPEAR_OK;
}

int device_info(DeviceInfo* out) {
  static std::mutex mu;
  static std::vector<DeviceInfo> cache;
  int dev = 0;
  if (int rc = cuda_check(cudaGetDevice(&dev), "cudaGetDevice")) return rc;
  std::lock_guard<std::mutex> lk(mu);
  for (const auto& d : cache)
    if (d.device == dev) { *out = d; return SPEAR_OK; }
  DeviceInfo d{};
  d.device = dev;
  int v = 0;
  if (int rc = cuda_check(cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev), "sm count")) return rc;
  if (int rc = cuda_check(cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev), "cc")) return rc;
  if (int rc = cuda_check(cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev), "cc")) return rc;
  if (int rc = cuda_check(cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev), "smem")) return rc;
  d.smem_optin = (size_t)v;
  if (d.cc_major != 10 || d.cc_minor != 3)
    return fail(SPEAR_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a only", dev,
                d.cc_major, d.cc_minor);
  cache.push_back(d);
  *out = d;
  return SPEAR_OK;
}

}  // namespace spear

using namespace spear;

extern "C" {

spear_status spear_pack_w4_sizes(int N, int K, int group_size, int symmetric, size_t* qweight_bytes,
                                 size_t* scales_bytes, size_t* zeros_bytes) {
  if (int rc = check_shape(N, K, group_size)) return rc;
  if (!qweight_bytes || !scales_bytes || !zeros_bytes) return fail(SPEAR_ERR_INVALID_ARG, "NULL size pointer");
  const size_t ng = (size_t)K / group_size;
  *qweight_bytes = (size_t)N * K / 2;
  *scales_bytes = (size_t)N * ng * 2;
  *zeros_bytes = symmetric ? 0 : (size_t)N * ((ng + 1) / 2);
  return SPEAR_OK;
}

spear_status spear_pack_w4(const float* W, int N, int K, int group_size, int symmetric, uint8_t* qweight,
                           uint16_t* scales, uint8_t* zeros, void* stream) {
  if (int rc = check_shape(N, K, group_size)) return rc;
  if (!W || !qweight || !scales || (!symmetric && !zeros)) return fail(SPEAR_ERR_INVALID_ARG, "NULL buffer");
  if (!aligned16(W) || !aligned16(qweight) || !aligned16(scales) || (zeros && !aligned16(zeros)))
    return fail(SPEAR_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
  DeviceInfo di;
  if (int rc = device_info(&di)) return rc;
  return launch_pack_w4(W, N, K, group_size, symmetric ? 1 : 0, qweight, scales, zeros,
                        static_cast<cudaStream_t>(stream));
}

spear_status spear_decode_workspace_bytes(const spear_w4_layer* L, int M, size_t* bytes) {
  if (int rc = check_layer(L)) return rc;
  if (M < 0 || M > 64) return fail(SPEAR_ERR_INVALID_ARG, "decode M=%d must be in [0, 64]", M);
  if (!bytes) return fail(SPEAR_ERR_INVALID_ARG, "bytes is NULL");
  if (M == 0) {                                      // an empty batch needs no workspace
    *bytes = 0;
    return SPEAR_OK;
  }
  return decode_workspace_bytes(*L, M, bytes);
}

spear_status spear_linear_decode(const spear_w4_layer* L, const uint16_t* x, int M, void* y, int out_dtype,
                                 void* workspace, size_t ws_bytes, void* stream) {
  if (int rc = check_layer(L)) return rc;
  if (M < 0 || M > 64) return fail(SPEAR_ERR_INVALID_ARG, "decode M=%d must be in [0, 64]", M);
  if (M == 0) return SPEAR_OK;                       // an empty batch: nothing to read or write
  if (!x || !y || !aligned16(x) || !aligned16(y)) return fail(SPEAR_ERR_INVALID_ARG, "x/y NULL or misaligned");
  if (out_dtype != SPEAR_OUT_BF16 && out_dtype != SPEAR_OUT_F32)
    return fail(SPEAR_ERR_INVALID_ARG, "out_dtype=%d", out_dtype);
  return launch_decode(*L, x, M, y, out_dtype == SPEAR_OUT_F32, workspace, ws_bytes,
                       static_cast<cudaStream_t>(stream), launch_overlap());
}

spear_status spear_linear_decode_noalloc(const spear_w4_layer* L, const uint16_t* x, int M, void* y,
                                         int out_dtype, void* stream) {
  if (int rc = check_layer(L)) return rc;
  if (M < 0 || M > 64) return fail(SPEAR_ERR_INVALID_ARG, "decode M=%d must be in [0, 64]", M);
  if (M == 0) return SPEAR_OK;                       // an empty batch: nothing to read or write
  if (!x || !y || !aligned16(x) || !aligned16(y)) return fail(SPEAR_ERR_INVALID_ARG, "x/y NULL or misaligned");
  if (out_dtype != SPEAR_OUT_BF16 && out_dtype != SPEAR_OUT_F32)
    return fail(SPEAR_ERR_INVALID_ARG, "out_dtype=%d", out_dtype);
  return launch_decode_noalloc(*L, x, M, y, out_dtype == SPEAR_OUT_F32, static_cast<cudaStream_t>(stream));
}

spear_status spear_prefill_workspace_bytes(const spear_w4_layer* L, int M, int mode, size_t* bytes) {
  if (int rc = check_layer(L)) return rc;
  if (M < 0) return fail(SPEAR_ERR_INVALID_ARG, "prefill M=%d must not be negative", M);
  if (mode < SPEAR_PREFILL_AUTO || mode > SPEAR_PREFILL_STREAM) return fail(SPEAR_ERR_INVALID_ARG, "mode=%d", mode);
  if (!bytes) return fail(SPEAR_ERR_INVALID_ARG, "bytes is NULL");
  if (M == 0) {
    *bytes = 0;
    return SPEAR_OK;
  }
  return prefill_workspace_bytes(*L, M, mode, bytes);
}

spear_status spear_linear_prefill(const spear_w4_layer* L, const uint16_t* x, int M, void* y, int out_dtype,
                                  int mode, void* workspace, size_t ws_bytes, void* stream, void* stream_aux) {
  if (int rc = check_layer(L)) return rc;
  if (M < 0) return fail(SPEAR_ERR_INVALID_ARG, "prefill M=%d must not be negative", M);
  if (mode < SPEAR_PREFILL_AUTO || mode > SPEAR_PREFILL_STREAM) return fail(SPEAR_ERR_INVALID_ARG, "mode=%d", mode);
  if (M == 0) return SPEAR_OK;                       // an empty batch: nothing to read or write
  if (!x || !y || !aligned16(x) || !aligned16(y)) return fail(SPEAR_ERR_INVALID_ARG, "x/y NULL or misaligned");
  if (out_dtype != SPEAR_OUT_BF16 && out_dtype != SPEAR_OUT_F32)
    return fail(SPEAR_ERR_INVALID_ARG, "out_dtype=%d", out_dtype);
  if (mode < SPEAR_PREFILL_AUTO || mode > SPEAR_PREFILL_STREAM) return fail(SPEAR_ERR_INVALID_ARG, "mode=%d", mode);
  return launch_prefill(*L, x, M, y, out_dtype == SPEAR_OUT_F32, mode, workspace, ws_bytes,
                        static_cast<cudaStream_t>(stream), static_cast<cudaStream_t>(stream_aux));
}

spear_status spear_workspace_init(void* workspace, size_t bytes, void* stream) {
  if (!workspace && bytes) return fail(SPEAR_ERR_INVALID_ARG, "workspace is NULL");
  if (!bytes) return SPEAR_OK;
  return cuda_check(cudaMemsetAsync(workspace, 0, bytes, static_cast<cudaStream_t>(stream)), "workspace init");
}

// Module selection, host only (see spear.h).  Ranks modules by damage share
// per unit of relative cost, keeps round(exp(entropy)) of them and gives them
// one common rank, a multiple of 16, that fits the byte budget.
namespace {
// Latency of one curve at M: piecewise linear through the points, continued
// past either end along the two nearest points.
bool curve_ok(const spear_latency_curve& c) {
  if (c.n < 1 || !c.M || !c.us) return false;
  for (int i = 0; i < c.n; ++i) {
    if (!std::isfinite(c.us[i]) || c.us[i] < 0.0f) return false;
    if (i > 0 && c.M[i] <= c.M[i - 1]) return false;
  }
  return true;
}
double curve_at(const spear_latency_curve& c, double M) {
  if (c.n == 1) return c.us[0];
  int i = 0;                                        // segment [i, i + 1]
  while (i + 2 < c.n && M > c.M[i + 1]) ++i;
  const double m0 = c.M[i], m1 = c.M[i + 1], u0 = c.us[i], u1 = c.us[i + 1];
  return u0 + (u1 - u0) * (M - m0) / (m1 - m0);
}
}  // namespace

spear_status spear_chunk_select(const spear_latency_curve* prefill, const spear_latency_curve* decode,
                                int nlayers, int decode_tokens, const int* choices, int nchoices,
                                double itl_target_us, int* chunk_out, double* step_us_out) {
  if (!prefill || !decode || nlayers <= 0 || !choices || nchoices <= 0 || !chunk_out || decode_tokens < 0 ||
      !(itl_target_us >= 0.0))
    return spear::fail(SPEAR_ERR_INVALID_ARG, "chunk_select: bad arguments");
  for (int l = 0; l < nlayers; ++l)
    if (!curve_ok(prefill[l]) || !curve_ok(decode[l]))
      return spear::fail(SPEAR_ERR_INVALID_ARG, "chunk_select: curve of layer %d invalid", l);
  for (int i = 0; i < nchoices; ++i)
    if (choices[i] < 0) return spear::fail(SPEAR_ERR_INVALID_ARG, "chunk_select: choices[%d] < 0", i);
  auto step = [&](int C) {
    double s = 0.0;
    if (C > 0) {
      for (int l = 0; l < nlayers; ++l) s += curve_at(prefill[l], (double)C + decode_tokens);
    } else if (decode_tokens > 0) {
      for (int l = 0; l < nlayers; ++l) s += curve_at(decode[l], (double)decode_tokens);
    }
    return s;
  };
  int best = -1, smallest = choices[0];
  for (int i = 0; i < nchoices; ++i) {
    smallest = std::min(smallest, choices[i]);
    if (step(choices[i]) <= itl_target_us && choices[i] > best) best = choices[i];
  }
  const int C = best >= 0 ? best : smallest;
  *chunk_out = C;
  if (step_us_out) *step_us_out = step(C);
  return SPEAR_OK;
}

spear_status spear_layer_select_mask(const float* damage, const float* cost, int L, double budget_bytes,
                                     int rank_min, int rank_max, uint8_t* mask_out, int* rank_out) {
  if (!damage || !cost || !mask_out || !rank_out || L <= 0) return fail(SPEAR_ERR_INVALID_ARG, "bad arguments");
  if (rank_min <= 0 || rank_max < rank_min || !(budget_bytes >= 0.0))
    return fail(SPEAR_ERR_INVALID_ARG, "rank range [%d, %d] or budget invalid", rank_min, rank_max);
  const int rank_lo = (rank_min + 15) / 16 * 16, rank_hi = rank_max / 16 * 16;
  if (rank_lo > rank_hi) return fail(SPEAR_ERR_INVALID_ARG, "no multiple of 16 in [%d, %d]", rank_min, rank_max);
  double total_damage = 0.0, total_cost = 0.0;
  for (int i = 0; i < L; ++i) {
    if (!std::isfinite(damage[i]) || damage[i] < 0.0f) return fail(SPEAR_ERR_INVALID_ARG, "damage[%d] invalid", i);
    if (!std::isfinite(cost[i]) || cost[i] <= 0.0f) return fail(SPEAR_ERR_INVALID_ARG, "cost[%d] invalid", i);
    total_damage += damage[i];
    total_cost += cost[i];
  }
  std::fill(mask_out, mask_out + L, 0);
  std::fill(rank_out, rank_out + L, 0);
  if (total_damage <= 0.0) return SPEAR_OK;

  double entropy = 0.0;
  std::vector<double> share(L), score(L);
  const double mean_cost = total_cost / L;
  for (int i = 0; i < L; ++i) {
    share[i] = damage[i] / total_damage;
    if (share[i] > 0.0) entropy -= share[i] * std::log(share[i]);
    score[i] = share[i] / (cost[i] / mean_cost);
  }
  int keep = (int)std::floor(std::exp(entropy) + 0.5);
  keep = std::min(std::max(keep, 1), L);
  std::vector<int> order(L);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return score[a] > score[b]; });

  for (; keep >= 1; --keep) {
    double used = 0.0;
    for (int i = 0; i < keep; ++i) used += cost[order[i]];
    int rank = 0;
    for (int r = rank_hi; r >= rank_lo; r -= 16)
      if ((double)r * used <= budget_bytes) { rank = r; break; }
    if (rank) {
      for (int i = 0; i < keep; ++i) { mask_out[order[i]] = 1; rank_out[order[i]] = rank; }
      return SPEAR_OK;
    }
  }
  return SPEAR_OK;
}

spear_status spear_set_wait_limit_ns(uint64_t ns) {
  spear::g_wait_limit_ns.store(ns);
  return SPEAR_OK;
}

spear_status spear_set_launch_overlap(int enable) {
  spear::set_launch_overlap(enable != 0);
  return SPEAR_OK;
}

spear_status spear_get_device_status(int* out, void* stream) {
  if (!out) return fail(SPEAR_ERR_INVALID_ARG, "out is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned s_pack = 0, s_dec = 0, s_pre = 0;
  if (int rc = read_and_clear_status_pack(&s_pack, st)) return rc;
  unsigned s_dtc = 0, s_dks = 0, s_dtm = 0;
  if (int rc = read_and_clear_status_decode(&s_dec, st)) return rc;
  if (int rc = read_and_clear_status_decode_tc(&s_dtc, st)) return rc;
  if (int rc = read_and_clear_status_decode_ks(&s_dks, st)) return rc;
  if (int rc = read_and_clear_status_decode_tm(&s_dtm, st)) return rc;
  if (!s_dec) s_dec = s_dtm ? s_dtm : s_dks ? s_dks : s_dtc;
  if (int rc = read_and_clear_status_prefill(&s_pre, st)) return rc;
  if (int rc = cuda_check(cudaStreamSynchronize(st), "status sync")) return rc;
  *out = (int)(s_pack ? s_pack : s_dec ? s_dec : s_pre);
  return SPEAR_OK;
}

const char* spear_status_string(int status) {
  switch (status) {
    case SPEAR_OK: return "SPEAR_OK";
    case SPEAR_ERR_INVALID_ARG: return "SPEAR_ERR_INVALID_ARG";
    case SPEAR_ERR_UNSUPPORTED: return "SPEAR_ERR_UNSUPPORTED";
    case SPEAR_ERR_WORKSPACE: return "SPEAR_ERR_WORKSPACE";
    case SPEAR_ERR_CUDA: return "SPEAR_ERR_CUDA";
    case SPEAR_ERR_TIMEOUT: return "SPEAR_ERR_TIMEOUT";
    case SPEAR_ERR_BOUNDS: return "SPEAR_ERR_BOUNDS";
    default: return "SPEAR_ERR_UNKNOWN";
  }
}

const char* spear_last_error(void) { return t_last_error; }

const char* spear_version(void) { return "0.1.0"; }

}  // extern "C"
