// pack.cu -- round-to-nearest int4 quantisation and nibble packing on the GPU
// (SPEAR explainer, Technical Summary 3.1: RTN W4, per-channel or grouped).
//
// One warp per (row n, pair of groups).  Per group of G consecutive k:
//   symmetric : s = fp16_ru(max|w| / 7),           u = clamp(rint(w/s), -8, 7) + 8
//   asymmetric: s = fp16_ru((hi - lo) / 15) with lo = min(min w, 0), hi = max(max w, 0),
//               z = clamp(rint(-lo/s), 0, 15),      u = clamp(rint(w/s) + z, 0, 15)
// All divisions are IEEE fp32 round-to-nearest (__fdiv_rn) and rint is
// round-half-to-even (__float2int_rn), so the bytes match any other correct
// implementation of the same definition bit for bit.  The max/min reductions
// are exact in any order.
//
// HBM-bound: reads 4 bytes per weight (twice: the range pass and the code
// pass; the second pass mostly hits L2), writes half a byte.
#include "common.cuh"
#include "internal.h"

namespace spear {
namespace {

__device__ unsigned g_pack_status;

constexpr int kPackWarps = 8;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Quantises group gi of row `w` (G floats starting at k0) and writes its codes;
// returns the zero point (8 for symmetric).  Lanes walk the group in chunks
// of 8 consecutive weights (two float4 loads, one 32-bit store of codes).
__device__ int quantize_group(const float* __restrict__ w, int k0, int G, int sym,
                              uint8_t* __restrict__ qrow, __half* __restrict__ scale_out, int lane) {
  const int nch = G / 8;
  float lo = 0.0f, hi = 0.0f, amax = 0.0f;
  bool finite = true;
  for (int j = lane; j < nch; j += 32) {
    const float4 a = *reinterpret_cast<const float4*>(w + k0 + 8 * j);
    const float4 b = *reinterpret_cast<const float4*>(w + k0 + 8 * j + 4);
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      finite = finite && isfinite(v[i]);
      lo = fminf(lo, v[i]);
      hi = fmaxf(hi, v[i]);
      amax = fmaxf(amax, fabsf(v[i]));
    }
  }
  finite = __all_sync(0xffffffffu, finite);
  lo = warp_min(lo);
  hi = warp_max(hi);
  amax = warp_max(amax);

  const float s32 = sym ? __fdiv_rn(amax, 7.0f) : __fdiv_rn(hi - lo, 15.0f);
  __half s16 = __float2half_ru(s32);
  const float s = __half2float(s16);
  if (!finite || isinf(s)) {
    if (lane == 0) record_status(&g_pack_status, DEV_ERR_INVALID);
    s16 = __float2half_rn(0.0f);
  }
  if (lane == 0) *scale_out = s16;
  const bool zero_group = !(s > 0.0f) || !finite || isinf(s);
  int z = 8;
  if (!sym) z = zero_group ? 0 : min(max(__float2int_rn(__fdiv_rn(-lo, s)), 0), 15);

  for (int j = lane; j < nch; j += 32) {
    const float4 a = *reinterpret_cast<const float4*>(w + k0 + 8 * j);
    const float4 b = *reinterpret_cast<const float4*>(w + k0 + 8 * j + 4);
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t packed = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int u;
      if (zero_group) {
        u = z;
      } else if (sym) {
        u = min(max(__float2int_rn(__fdiv_rn(v[i], s)), -8), 7) + 8;
      } else {
        u = min(max(__float2int_rn(__fdiv_rn(v[i], s)) + z, 0), 15);
      }
      packed |= (uint32_t)u << (4 * i);
    }
    *reinterpret_cast<uint32_t*>(qrow + (k0 + 8 * j) / 2) = packed;
  }
  return z;
}

__global__ void __launch_bounds__(32 * kPackWarps)
pack_w4_kernel(const float* __restrict__ W, int N, int K, int G, int sym, uint8_t* __restrict__ qweight,
               __half* __restrict__ scales, uint8_t* __restrict__ zeros) {
  const int lane = threadIdx.x & 31;
  const int ng = K / G;
  const int npairs = (ng + 1) / 2;
  const long long item = (long long)blockIdx.x * kPackWarps + (threadIdx.x >> 5);
  if (item >= (long long)N * npairs) return;
  const int n = (int)(item / npairs);
  const int pair = (int)(item % npairs);
  const float* w = W + (size_t)n * K;
  uint8_t* qrow = qweight + (size_t)n * (K / 2);
  int zbyte = 0;
#pragma unroll 1
  for (int h = 0; h < 2; ++h) {
    const int gi = 2 * pair + h;
    if (gi >= ng) break;
    SPEAR_CHECK(&g_pack_status, n < N && gi * G + G <= K && (gi * G) % 2 == 0);
    const int z = quantize_group(w, gi * G, G, sym, qrow, scales + (size_t)n * ng + gi, lane);
    zbyte |= z << (4 * h);
  }
  if (!sym && lane == 0) zeros[(size_t)n * npairs + pair] = (uint8_t)zbyte;
}

}  // namespace

int launch_pack_w4(const float* W, int N, int K, int G, int sym, uint8_t* qweight, uint16_t* scales,
                   uint8_t* zeros, cudaStream_t st) {
  const long long items = (long long)N * ((K / G + 1) / 2);
  const long long blocks = (items + kPackWarps - 1) / kPackWarps;
  if (blocks > 0x7fffffffLL) return fail(SPEAR_ERR_UNSUPPORTED, "pack: %d x %d is too large", N, K);
  pack_w4_kernel<<<(unsigned)blocks, 32 * kPackWarps, 0, st>>>(W, N, K, G, sym, qweight,
                                                               reinterpret_cast<__half*>(scales), zeros);
  return cuda_check(cudaGetLastError(), "pack_w4 launch");
}

int read_and_clear_status_pack(unsigned* out, cudaStream_t st) {
  void* addr = nullptr;
  if (int rc = cuda_check(cudaGetSymbolAddress(&addr, g_pack_status), "pack status address")) return rc;
  if (int rc = cuda_check(cudaMemcpyAsync(out, addr, sizeof(unsigned), cudaMemcpyDeviceToHost, st), "read pack status")) return rc;
  if (int rc = cuda_check(cudaStreamSynchronize(st), "read pack status")) return rc;
  return cuda_check(cudaMemsetAsync(addr, 0, sizeof(unsigned), st), "clear pack status");
}

}  // namespace spear
