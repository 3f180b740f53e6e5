// decode.cu -- fused decode kernel for the gated W4 + low-rank compensated
// linear (SPEAR explainer, Technical Summary 2.2 A: in the memory-bound decode
// phase the compensator is fused into the low-bit GEMM epilogue so the layer
// is ONE kernel launch).
//
//   y[m][n] = sum_k (u[n][k] - z[n][g]) s[n][g] x[m][k]  +  alpha g_m sum_j B[n][j] t_m[j]
//   t_m = A x_m,  g_m = sigmoid(w_g . x_m + b_g)
//
// Design (one cooperative launch, every thread block resident):
//  * Producer blocks (the first Q) compute the rank-(r+1) down-projection
//    P = [A; w_g] x over disjoint K slices with bf16 mma.sync, write their
//    slice partials to the workspace, and the last producer to arrive sums
//    them in a fixed order, applies the gate and publishes T = alpha g t with
//    a release flag.
//  * Streamer blocks split the (16-row tile x 128-k chunk) work items of the
//    int4 weight evenly ("stream-K"): each block owns one contiguous range,
//    so every SM streams the same number of weight bytes.  Weights move
//    global -> shared through a per-warp cp.async ring (L1 bypass), are turned
//    into exact small integers in registers (nibble | bf16 bias, minus the
//    biased zero point) and multiplied by the tokens with mma.sync; the group
//    scale is applied to each 128-k partial in fp32.  A tile split across two
//    blocks is finished by whichever block arrives last (fixed-order sum of
//    the parts from the workspace).
//  * Only the epilogue depends on T: each streamer waits (bounded) for the
//    flag after all of its weight traffic, adds B T with one more small mma,
//    and stores y.  The last streamer resets the flag, so the workspace's
//    synchronisation words are zero again between calls.
//
// HBM traffic per call: N K / 2 (codes) + N K/G * 2 (scales) + zeros + (r+1) K 2
// (A, w_g) + N r 2 (B) + M K 2 (x) + M N 2 (y): the roofline of this kernel.
#include <algorithm>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace spear {
namespace {

__device__ unsigned g_decode_status;

constexpr int kThreads = 256;
constexpr int kWarps = 8;
constexpr int kStages = 6;            // cp.async ring depth per warp (1 KB per stage)
constexpr int kChunkK = 128;          // k per work item
constexpr int kMaxRank = 64;
constexpr unsigned long long kWaitLimitNs = 200ull * 1000 * 1000;   // 200 ms

struct DecodeParams {
  int N, K, G, M, sym;
  const uint8_t* qweight;
  const __half* scales;
  const uint8_t* zeros;
  const __nv_bfloat16* x;
  void* y;
  int out_f32;
  int r;
  const __nv_bfloat16* A;
  const __nv_bfloat16* B;
  const __nv_bfloat16* w_g;
  float b_g, alpha;
  // work split
  int Q, P;                 // producer / streamer blocks
  int tiles, nchunks;       // N/16, K/128
  long long units;          // tiles * nchunks
  int max_tiles;            // most tiles one streamer touches
  int max_parts;            // most streamers sharing one tile
  int ng;                   // K/G
  // workspace
  float* ws_prod;           // [Q][Mpad][16]
  float* ws_T;              // [Mpad][r]
  float* ws_part;           // [tiles][max_parts][MT*4*32]
  unsigned* ws_tile_cnt;    // [tiles]
  unsigned* ws_sync;        // [0] producer ticket, [1] T flag, [2] streamer ticket
};

__device__ __forceinline__ long long unit_begin(long long b, long long U, int P) { return b * U / P; }
__device__ __forceinline__ int unit_owner(long long u, long long U, int P) {
  return (int)(((u + 1) * P + U - 1) / U - 1);
}

// ---------------------------------------------------------------- producer --
// Producer block q computes the partial P[m][i] = sum_{k in slice s} W'[i][k] x[m][k]
// for one 16-row tile rt = q % RT of W' = [A; w_g; 0-padding] over K slice
// s = q / RT (S = Q / RT slices), so its loads take one round trip.
// Lane (g, c) of a warp loads 16 B (8 consecutive k) per row; within a 32-k
// piece the MMA's k positions {2c, 2c+1, 2c+8, 2c+9} of k-step h map to the
// lane's k = 8c + 4h + {0, 1, 2, 3}, identically for both operands.
constexpr int kMaxSlices = 8;

template <int MT>
__device__ void producer_block(const DecodeParams& p, float* smem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int RT = (p.r + 1 + 15) / 16;
  const int Mpad = MT * 8;
  const int q = blockIdx.x, rt = q % RT, sl = q / RT, S = p.Q / RT;
  const int c0 = (int)((long long)sl * p.nchunks / S), c1 = (int)((long long)(sl + 1) * p.nchunks / S);
  const int npieces = (c1 - c0) * 4;                   // 32-k pieces of the slice
  float* red = smem;                                   // [kWarps][MT][4][32]

  auto row_ptr = [&](int i) -> const __nv_bfloat16* {
    if (i < p.r) return p.A + (size_t)i * p.K;
    if (i == p.r) return p.w_g;
    return nullptr;
  };
  const __nv_bfloat16* wlo = row_ptr(rt * 16 + g);
  const __nv_bfloat16* whi = row_ptr(rt * 16 + g + 8);
  float acc[MT][4];
#pragma unroll
  for (int t = 0; t < MT; ++t)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[t][i] = 0.0f;
  for (int pc0 = warp; pc0 < npieces; pc0 += 2 * kWarps) {
    // two pieces per pass: all of their loads are in flight together
    uint4 va[2], vb[2], xv[2][MT];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int pc = pc0 + h * kWarps;
      const bool ok = pc < npieces;
      const int kb = c0 * kChunkK + pc * 32 + 8 * c;
      va[h] = (ok && wlo) ? ldg16(wlo + kb) : make_uint4(0, 0, 0, 0);
      vb[h] = (ok && whi) ? ldg16(whi + kb) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        const int tok = t * 8 + g;
        xv[h][t] = (ok && tok < p.M) ? ldg16(p.x + (size_t)tok * p.K + kb) : make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        mma_bf16_16816(acc[t], va[h].x, vb[h].x, va[h].y, vb[h].y, xv[h][t].x, xv[h][t].y);
        mma_bf16_16816(acc[t], va[h].z, vb[h].z, va[h].w, vb[h].w, xv[h][t].z, xv[h][t].w);
      }
  }
  // cross-warp sum in a fixed order; this block's partial for its 16 rows
#pragma unroll
  for (int t = 0; t < MT; ++t)
#pragma unroll
    for (int i = 0; i < 4; ++i) red[((warp * MT + t) * 4 + i) * 32 + lane] = acc[t][i];
  __syncthreads();
  for (int e = threadIdx.x; e < MT * 4 * 32; e += kThreads) {
    const int t = e / 128, i = (e / 32) & 3, ln = e & 31;
    float v = 0.0f;
    for (int w = 0; w < kWarps; ++w) v += red[((w * MT + t) * 4 + i) * 32 + ln];
    // C fragment element i of lane ln: row (ln/4) + 8 (i/2), token t*8 + 2 (ln%4) + (i%2)
    const int row = (ln >> 2) + 8 * (i >> 1);
    const int tok = t * 8 + 2 * (ln & 3) + (i & 1);
    p.ws_prod[((size_t)q * Mpad + tok) * 16 + row] = v;
    __threadfence();
  }
  __syncthreads();

  // arrive; the last producer sums the slices, applies the gate, publishes T
  __shared__ unsigned s_last;
  if (threadIdx.x == 0) {
    const unsigned old = atomicAdd(&p.ws_sync[0], 1u);
    s_last = (old == (unsigned)(p.Q - 1));
    __threadfence();
  }
  __syncthreads();
  if (!s_last) return;
  auto slice_sum = [&](int m, int i) {                  // fixed order over slices
    const int rti = i / 16, ri = i % 16;
    float part[kMaxSlices];
#pragma unroll
    for (int ss = 0; ss < kMaxSlices; ++ss)
      part[ss] = ss < S ? __ldcg(p.ws_prod + ((size_t)(ss * RT + rti) * Mpad + m) * 16 + ri) : 0.0f;
    float v = 0.0f;
#pragma unroll
    for (int ss = 0; ss < kMaxSlices; ++ss) v += part[ss];
    return v;
  };
  float* gate = smem;                                   // [Mpad]
  for (int m = threadIdx.x; m < Mpad; m += kThreads) gate[m] = 1.0f / (1.0f + expf(-(slice_sum(m, p.r) + p.b_g)));
  __syncthreads();
  for (int e = threadIdx.x; e < Mpad * p.r; e += kThreads) {
    const int m = e / p.r, j = e % p.r;
    const float v = slice_sum(m, j);
    p.ws_T[e] = (m < p.M) ? p.alpha * gate[m] * v : 0.0f;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    p.ws_sync[0] = 0;                                   // ticket ready for the next call
    st_release_gpu(&p.ws_sync[1], 1u);
  }
}

// ---------------------------------------------------------------- streamer --

// Work cursor of one warp over its items: (segment, chunk) with chunk stepping
// by kWarps inside [ca, cb) of each segment.
struct Cursor {
  int seg, ch;
};

template <int MT, bool COMP, bool PERCH>
__device__ void streamer_block(const DecodeParams& p, float* smem) {
  constexpr bool XPF = (MT == 1);                        // prefetch the next item's tokens in registers
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int b = blockIdx.x - p.Q;
  const long long u0 = unit_begin(b, p.units, p.P), u1 = unit_begin(b + 1, p.units, p.P);
  const int tile0 = (int)(u0 / p.nchunks);
  const int tile_last = u1 > u0 ? (int)((u1 - 1) / p.nchunks) : tile0 - 1;
  const int nseg = tile_last - tile0 + 1;                  // 0 for an empty range
  const int Mpad = MT * 8;
  const size_t half_k = (size_t)p.K / 2;

  // shared memory carve-up
  uint4* ring = reinterpret_cast<uint4*>(smem);                       // [kWarps][kStages][2][32]
  float* red = smem + kWarps * kStages * 2 * 32 * 4;                  // [kWarps][MT][4][32]
  float* ybuf = red + kWarps * MT * 4 * 32;                           // [max_tiles][MT][4][32]
  uint32_t* Ts = reinterpret_cast<uint32_t*>(ybuf + p.max_tiles * MT * 4 * 32);  // [Mpad][r/2] hi, then lo
  __half* sc_s = reinterpret_cast<__half*>(Ts + (COMP ? Mpad * kMaxRank : 0));   // [max_tiles][16][ng]
  uint8_t* z_s = reinterpret_cast<uint8_t*>(sc_s + p.max_tiles * 16 * p.ng);     // [max_tiles][16][ng]
  __shared__ int s_parts[64];      // streamers sharing the segment's tile (1 = this block owns it)
  __shared__ int s_fixup[64];      // 1 when this block stores the segment's tile
  __shared__ int s_flag;

  auto seg_ca = [&](int s) {
    return (int)(max(u0, (long long)(tile0 + s) * p.nchunks) - (long long)(tile0 + s) * p.nchunks);
  };
  auto seg_cb = [&](int s) {
    return (int)(min(u1, (long long)(tile0 + s + 1) * p.nchunks) - (long long)(tile0 + s) * p.nchunks);
  };

  // per-warp item cursor over the segments
  auto first_item = [&](Cursor& cur) {
    cur.seg = 0;
    cur.ch = nseg > 0 ? seg_ca(0) + warp : 0;
    while (cur.seg < nseg && cur.ch >= seg_cb(cur.seg)) {
      ++cur.seg;
      if (cur.seg < nseg) cur.ch = seg_ca(cur.seg) + warp;
    }
  };
  auto next_item = [&](Cursor& cur) {
    cur.ch += kWarps;
    while (cur.seg < nseg && cur.ch >= seg_cb(cur.seg)) {
      ++cur.seg;
      if (cur.seg < nseg) cur.ch = seg_ca(cur.seg) + warp;
    }
  };
  uint4* my_ring = ring + warp * kStages * 2 * 32;
  auto issue = [&](const Cursor& cur, int slot) {
    if (cur.seg < nseg) {
      const int n0 = (tile0 + cur.seg) * 16;
      const uint8_t* src = p.qweight + (size_t)(n0 + g) * half_k + (size_t)cur.ch * (kChunkK / 2) + c * 16;
      cp_async16(my_ring + (slot * 2 + 0) * 32 + lane, src);
      cp_async16(my_ring + (slot * 2 + 1) * 32 + lane, src + 8 * half_k);
    }
    cp_async_commit();
  };

  // 1. weight stream first
  Cursor icur, ccur;
  first_item(icur);
  ccur = icur;
#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    issue(icur, s);
    next_item(icur);
  }
  // 2. scales and zero points of every touched tile, loads batched ahead of the stores
  {
    const int total = nseg * 16 * p.ng;
    const int zrow = (p.ng + 1) / 2;
    for (int e0 = threadIdx.x; e0 < total; e0 += 8 * kThreads) {
      __half sv[8];
      uint8_t zv[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int e = e0 + u * kThreads;
        sv[u] = __ushort_as_half(0);
        zv[u] = 8;
        if (e < total) {
          const int sg = e / (16 * p.ng), rem = e % (16 * p.ng), row = rem / p.ng, gi = rem % p.ng;
          const int n = (tile0 + sg) * 16 + row;
          sv[u] = p.scales[(size_t)n * p.ng + gi];
          if (!p.sym) {
            const uint8_t zb = p.zeros[(size_t)n * zrow + gi / 2];
            zv[u] = (gi & 1) ? (zb >> 4) : (zb & 15);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int e = e0 + u * kThreads;
        if (e < total) { sc_s[e] = sv[u]; z_s[e] = zv[u]; }
      }
    }
  }
  // 3. tokens of the first item
  uint4 xcur[MT][4];
  auto load_x = [&](const Cursor& cur, uint4 (&dst)[MT][4]) {
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const int tok = t * 8 + g;
        dst[t][w] = (cur.seg < nseg && tok < p.M)
                        ? ldg16(p.x + (size_t)tok * p.K + (size_t)cur.ch * kChunkK + 32 * c + 8 * w)
                        : make_uint4(0, 0, 0, 0);
      }
  };
  if (XPF) load_x(ccur, xcur);
  int slot = 0;
  __syncthreads();                                      // scales staged

  for (int seg = 0; seg < nseg; ++seg) {
    const int tile = tile0 + seg;
    float acc[MT][4];
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[t][i] = 0.0f;

    while (ccur.seg == seg) {
      issue(icur, (slot + kStages - 1) % kStages);
      next_item(icur);
      Cursor nx = ccur;
      next_item(nx);
      uint4 xnext[MT][4];
      if (XPF) load_x(nx, xnext);                        // in flight while this item computes
      else load_x(ccur, xcur);
      cp_async_wait<kStages - 1>();
      const uint4 wlo = my_ring[(slot * 2 + 0) * 32 + lane];
      const uint4 whi = my_ring[(slot * 2 + 1) * 32 + lane];
      const int ch = ccur.ch;
      const int gi = ch * kChunkK / p.G;
      const int srow = seg * 16 * p.ng;
      const uint32_t zlo = bf16x2_bias(z_s[srow + g * p.ng + gi]);
      const uint32_t zhi = bf16x2_bias(z_s[srow + (g + 8) * p.ng + gi]);
      float part[MT][4];
#pragma unroll
      for (int t = 0; t < MT; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) part[t][i] = 0.0f;
      const uint32_t wl[4] = {wlo.x, wlo.y, wlo.z, wlo.w};
      const uint32_t wh[4] = {whi.x, whi.y, whi.z, whi.w};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t va[4], vb[4];
        nibbles_to_bf16x2_biased(wl[w], va);
        nibbles_to_bf16x2_biased(wh[w], vb);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          va[i] = bf16x2_sub(va[i], zlo);                // exact (u - z)
          vb[i] = bf16x2_sub(vb[i], zhi);
        }
#pragma unroll
        for (int t = 0; t < MT; ++t) {
          const uint4 xv = xcur[t][w];
          // k positions: step 0 pairs nibbles (0,4),(1,5); step 1 pairs (2,6),(3,7)
          const uint32_t b00 = __byte_perm(xv.x, xv.z, 0x5410), b01 = __byte_perm(xv.x, xv.z, 0x7632);
          const uint32_t b10 = __byte_perm(xv.y, xv.w, 0x5410), b11 = __byte_perm(xv.y, xv.w, 0x7632);
          mma_bf16_16816(part[t], va[0], vb[0], va[1], vb[1], b00, b01);
          mma_bf16_16816(part[t], va[2], vb[2], va[3], vb[3], b10, b11);
        }
      }
      if (PERCH) {
#pragma unroll
        for (int t = 0; t < MT; ++t)
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[t][i] += part[t][i];
      } else {
        const float slo = __half2float(sc_s[srow + g * p.ng + gi]);
        const float shi = __half2float(sc_s[srow + (g + 8) * p.ng + gi]);
#pragma unroll
        for (int t = 0; t < MT; ++t) {
          acc[t][0] = fmaf(slo, part[t][0], acc[t][0]);
          acc[t][1] = fmaf(slo, part[t][1], acc[t][1]);
          acc[t][2] = fmaf(shi, part[t][2], acc[t][2]);
          acc[t][3] = fmaf(shi, part[t][3], acc[t][3]);
        }
      }
      if (XPF) {
#pragma unroll
        for (int t = 0; t < MT; ++t)
#pragma unroll
          for (int w = 0; w < 4; ++w) xcur[t][w] = xnext[t][w];
      }
      ccur = nx;
      slot = (slot + 1) % kStages;
    }

    // ---- segment done: fixed-order sum over warps into ybuf (whole tile) or
    // this block's part of a shared tile (workspace; finished at the end)
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
      for (int i = 0; i < 4; ++i) red[((warp * MT + t) * 4 + i) * 32 + lane] = acc[t][i];
    __syncthreads();
    const long long tu0 = (long long)tile * p.nchunks, tu1 = tu0 + p.nchunks;
    const int first = unit_owner(tu0, p.units, p.P), last = unit_owner(tu1 - 1, p.units, p.P);
    const int parts = last - first + 1;
    float* dst = (parts == 1) ? ybuf + seg * MT * 128
                              : p.ws_part + ((size_t)tile * p.max_parts + (b - first)) * MT * 128;
    for (int e = threadIdx.x; e < MT * 128; e += kThreads) {
      float v = 0.0f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) v += red[w * MT * 128 + e];
      dst[e] = v;
    }
    if (threadIdx.x == 0) s_parts[seg] = parts;
    __syncthreads();
  }
  cp_async_wait<0>();

  // ---- one synchronisation point for every shared tile: arrive, and the
  // last block to arrive sums the parts (fixed order) and stores the tile
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int seg = 0; seg < nseg; ++seg) {
      if (s_parts[seg] == 1) { s_fixup[seg] = 1; continue; }
      const int tile = tile0 + seg;
      const unsigned old = atomicAdd(&p.ws_tile_cnt[tile], 1u);
      const int lastp = old == (unsigned)(s_parts[seg] - 1);
      if (lastp) p.ws_tile_cnt[tile] = 0;               // every part has arrived
      s_fixup[seg] = lastp;
    }
    __threadfence();
  }
  __syncthreads();
  for (int seg = 0; seg < nseg; ++seg) {
    if (s_parts[seg] == 1 || !s_fixup[seg]) continue;
    const float* src = p.ws_part + (size_t)(tile0 + seg) * p.max_parts * MT * 128;
    for (int e = threadIdx.x; e < MT * 128; e += kThreads) {
      float v = 0.0f;
      for (int pi = 0; pi < s_parts[seg]; ++pi) v += __ldcg(src + (size_t)pi * MT * 128 + e);
      ybuf[seg * MT * 128 + e] = v;
    }
  }

  // ---- the compensator's down-projection (published by the producers)
  if (COMP) {
    if (threadIdx.x == 0) {
      const uint64_t t0 = globaltimer_ns();
      unsigned ok = 0;
      for (unsigned it = 0;; ++it) {
        if (ld_acquire_gpu(&p.ws_sync[1])) { ok = 1; break; }
        if ((it & 63) == 63 && globaltimer_ns() - t0 > kWaitLimitNs) break;
        __nanosleep(32);
      }
      if (!ok) record_status(&g_decode_status, DEV_ERR_TIMEOUT);
      s_flag = ok;
    }
    __syncthreads();
    // T as bf16 hi + lo (T = hi + lo to ~2^-16 relative)
    for (int e = threadIdx.x; e < Mpad * p.r / 2; e += kThreads) {
      const int m = e / (p.r / 2), jj = (e % (p.r / 2)) * 2;
      float t0v = 0.0f, t1v = 0.0f;
      if (s_flag) {
        t0v = __ldcg(p.ws_T + m * p.r + jj);
        t1v = __ldcg(p.ws_T + m * p.r + jj + 1);
      }
      const __nv_bfloat16 h0 = __float2bfloat16_rn(t0v), h1 = __float2bfloat16_rn(t1v);
      Ts[m * (p.r / 2) + jj / 2] = pack_bf16x2(__bfloat162float(h0), __bfloat162float(h1));
      Ts[Mpad * (p.r / 2) + m * (p.r / 2) + jj / 2] =
          pack_bf16x2(t0v - __bfloat162float(h0), t1v - __bfloat162float(h1));
    }
  }
  __syncthreads();

  // ---- epilogue: y = acc (* per-channel scale) + B T, one (segment, token tile) per warp
  for (int item = warp; item < nseg * MT; item += kWarps) {
    const int seg = item / MT, t = item % MT;
    if (!s_fixup[seg]) continue;
    const int tile = tile0 + seg;
    const int n_lo = tile * 16 + g, n_hi = n_lo + 8;
    float v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = ybuf[(seg * MT + t) * 128 + i * 32 + lane];
    if (PERCH) {
      const float slo = __half2float(sc_s[seg * 16 * p.ng + g * p.ng]);
      const float shi = __half2float(sc_s[seg * 16 * p.ng + (g + 8) * p.ng]);
      v[0] *= slo; v[1] *= slo; v[2] *= shi; v[3] *= shi;
    }
    if (COMP) {
      const int rh = p.r / 2;
      for (int j0 = 0; j0 < p.r; j0 += 16) {
        const uint32_t* Blo = reinterpret_cast<const uint32_t*>(p.B + (size_t)n_lo * p.r + j0);
        const uint32_t* Bhi = reinterpret_cast<const uint32_t*>(p.B + (size_t)n_hi * p.r + j0);
        const uint32_t a0 = __ldg(Blo + c), a1 = __ldg(Bhi + c), a2 = __ldg(Blo + c + 4), a3 = __ldg(Bhi + c + 4);
        const int tok = t * 8 + g;
        const uint32_t* th = Ts + tok * rh + j0 / 2;
        const uint32_t* tl = Ts + Mpad * rh + tok * rh + j0 / 2;
        mma_bf16_16816(v, a0, a1, a2, a3, th[c], th[c + 4]);
        mma_bf16_16816(v, a0, a1, a2, a3, tl[c], tl[c + 4]);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int tok = t * 8 + 2 * c + (i & 1);
      const int n = (i < 2) ? n_lo : n_hi;
      if (tok < p.M) {
        if (p.out_f32) reinterpret_cast<float*>(p.y)[(size_t)tok * p.N + n] = v[i];
        else reinterpret_cast<__nv_bfloat16*>(p.y)[(size_t)tok * p.N + n] = __float2bfloat16_rn(v[i]);
      }
    }
  }

  if (COMP) {
    __syncthreads();
    if (threadIdx.x == 0) {
      const unsigned old = atomicAdd(&p.ws_sync[2], 1u);
      if (old == (unsigned)(p.P - 1)) {                 // every streamer is past its wait
        p.ws_sync[2] = 0;
        atomicExch(&p.ws_sync[1], 0u);
      }
    }
  }
}

template <int MT, bool COMP, bool PERCH>
__global__ void __launch_bounds__(kThreads, (MT <= 2 ? 2 : 1)) decode_kernel(const DecodeParams p) {
  extern __shared__ __align__(16) float smem[];
  if ((int)blockIdx.x < p.Q) {
    // The plain layer keeps the same block split as the compensated one (its
    // producer blocks idle), so forcing the gate to zero reproduces it bit for bit.
    if (COMP) producer_block<MT>(p, smem);
  } else {
    streamer_block<MT, COMP, PERCH>(p, smem);
  }
}

using KernelFn = void (*)(const DecodeParams);

template <int MT>
KernelFn pick_kernel(bool comp, bool perch) {
  if (comp) return perch ? decode_kernel<MT, true, true> : decode_kernel<MT, true, false>;
  return perch ? decode_kernel<MT, false, true> : decode_kernel<MT, false, false>;
}

KernelFn pick(int MT, bool comp, bool perch) {
  switch (MT) {
    case 1: return pick_kernel<1>(comp, perch);
    case 2: return pick_kernel<2>(comp, perch);
    case 4: return pick_kernel<4>(comp, perch);
    default: return pick_kernel<8>(comp, perch);
  }
}

int mt_for(int M) { return M <= 8 ? 1 : M <= 16 ? 2 : M <= 32 ? 4 : 8; }

// Host-side plan: block counts, the stream-K split and the workspace layout.
struct Plan {
  int device, N, K, G, rank, comp, MT;      // key
  int Q, P, tiles, nchunks, max_tiles, max_parts, ng, Rpad;
  long long units;
  size_t smem;
  size_t off_prod, off_T, off_part, off_cnt, off_sync, total;
  KernelFn fn;
};

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

size_t streamer_smem(int MT, bool comp, int max_tiles, int ng) {
  size_t s = (size_t)kWarps * kStages * 2 * 32 * 16;         // ring
  s += (size_t)kWarps * MT * 128 * 4;                        // red
  s += (size_t)max_tiles * MT * 128 * 4;                     // ybuf
  if (comp) s += (size_t)MT * 8 * kMaxRank * 4;              // T hi/lo
  s += (size_t)max_tiles * 16 * ng * 3;                      // scales + zeros
  return s;
}

int build_plan(const spear_w4_layer& L, int MT, bool comp, const DeviceInfo& di, Plan* pl) {
  const bool has_rank = L.rank > 0;          // the split depends on this, not on comp_enabled
  pl->MT = MT;
  pl->tiles = L.N / 16;
  pl->nchunks = L.K / kChunkK;
  pl->ng = L.K / L.group_size;
  pl->units = (long long)pl->tiles * pl->nchunks;
  pl->Rpad = ((L.rank + 1 + 15) / 16) * 16;
  const bool perch = L.group_size == L.K;
  pl->fn = pick(pl->MT, comp, perch);

  // The block count depends on occupancy, which depends on shared memory,
  // which depends on how many tiles one block touches: iterate to a fixed
  // point, then validate occupancy at the final size.
  int blocks = 2 * di.num_sms;
  bool settled = false;
  for (int iter = 0; iter < 8 && !settled; ++iter) {
    if (has_rank) {
      // RT row tiles x S K-slices; one slice's A bytes ~ one streamer's weight bytes
      const int RT = (L.rank + 1 + 15) / 16;
      const double w_per_block = (double)L.N * L.K / 2.0 / std::max(1, blocks - RT);
      const int S = (int)std::lround(32.0 * L.K / w_per_block);
      pl->Q = RT * std::max(1, std::min(S, std::min(kMaxSlices, pl->nchunks)));
    } else {
      pl->Q = 0;
    }
    pl->P = (int)std::max<long long>(1, std::min<long long>(blocks - pl->Q, pl->units));
    const long long per = std::max<long long>(1, pl->units / pl->P);   // floor of units per streamer
    pl->max_tiles = (int)std::min<long long>((per + pl->nchunks - 1) / pl->nchunks + 2, pl->tiles);
    pl->max_parts = (int)std::min<long long>((pl->nchunks + per - 1) / per + 1, pl->P);
    if (pl->max_tiles > 64) return fail(SPEAR_ERR_UNSUPPORTED, "decode: too many tiles per block");
    pl->smem = std::max(streamer_smem(pl->MT, has_rank, pl->max_tiles, pl->ng), (size_t)kWarps * pl->MT * 128 * 4);
    if (pl->smem > di.smem_optin)
      return fail(SPEAR_ERR_UNSUPPORTED, "decode: shape needs %zu B of shared memory", pl->smem);
    if (cudaFuncSetAttribute(pl->fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl->smem) != cudaSuccess)
      return fail(SPEAR_ERR_CUDA, "decode: cudaFuncSetAttribute failed");
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, pl->fn, kThreads, pl->smem) != cudaSuccess ||
        per_sm < 1)
      return fail(SPEAR_ERR_CUDA, "decode: occupancy query failed");
    const int cap = std::min(per_sm, 2) * di.num_sms;
    if (pl->Q + pl->P <= cap && (blocks == cap || pl->Q + pl->P < blocks)) settled = true;
    else blocks = cap;
  }
  if (!settled) return fail(SPEAR_ERR_UNSUPPORTED, "decode: no resident launch configuration");

  const int Mpad = pl->MT * 8;
  size_t off = 0;
  pl->off_sync = off; off = align256(off + 4 * sizeof(unsigned));
  pl->off_cnt = off;  off = align256(off + (size_t)pl->tiles * sizeof(unsigned));
  pl->off_prod = off; off = align256(off + (size_t)std::max(pl->Q, 1) * Mpad * 16 * 4);
  pl->off_T = off;    off = align256(off + (size_t)Mpad * std::max(L.rank, 1) * 4);
  pl->off_part = off; off = align256(off + (size_t)pl->tiles * pl->max_parts * pl->MT * 128 * 4);
  pl->total = off;
  return SPEAR_OK;
}

// Plans are cached per (device, shape, format, rank, compensator on/off, token
// tile count): the occupancy query and function attributes run once.
int get_plan(const spear_w4_layer& L, int M, Plan* out) {
  DeviceInfo di;
  if (int rc = device_info(&di)) return rc;
  const int MT = mt_for(M);
  const int comp = (L.comp_enabled && L.rank > 0) ? 1 : 0;
  static std::mutex mu;
  static std::vector<Plan> cache;
  std::lock_guard<std::mutex> lk(mu);
  for (const Plan& p : cache)
    if (p.device == di.device && p.N == L.N && p.K == L.K && p.G == L.group_size && p.rank == L.rank &&
        p.comp == comp && p.MT == MT) {
      *out = p;
      return SPEAR_OK;
    }
  Plan p{};
  if (int rc = build_plan(L, MT, comp != 0, di, &p)) return rc;
  p.device = di.device; p.N = L.N; p.K = L.K; p.G = L.group_size; p.rank = L.rank; p.comp = comp;
  if (cache.size() > 4096) cache.clear();
  cache.push_back(p);
  *out = p;
  return SPEAR_OK;
}

}  // namespace

int decode_workspace_bytes(const spear_w4_layer& L, int M, size_t* bytes) {
  Plan pl;
  if (int rc = get_plan(L, M, &pl)) return rc;
  *bytes = pl.total;
  return SPEAR_OK;
}

int launch_decode(const spear_w4_layer& L, const uint16_t* x, int M, void* y, int out_f32, void* ws,
                  size_t ws_bytes, cudaStream_t st) {
  Plan pl;
  if (int rc = get_plan(L, M, &pl)) return rc;
  if (!ws || ws_bytes < pl.total)
    return fail(SPEAR_ERR_WORKSPACE, "decode: workspace of %zu B is smaller than the %zu B needed", ws_bytes, pl.total);
  if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0)
    return fail(SPEAR_ERR_INVALID_ARG, "decode: workspace must be 256-byte aligned");
  DecodeParams p{};
  p.N = L.N; p.K = L.K; p.G = L.group_size; p.M = M; p.sym = L.symmetric;
  p.qweight = L.qweight;
  p.scales = reinterpret_cast<const __half*>(L.scales);
  p.zeros = L.zeros;
  p.x = reinterpret_cast<const __nv_bfloat16*>(x);
  p.y = y; p.out_f32 = out_f32;
  p.r = pl.comp ? L.rank : 0;
  p.A = reinterpret_cast<const __nv_bfloat16*>(L.A);
  p.B = reinterpret_cast<const __nv_bfloat16*>(L.B);
  p.w_g = reinterpret_cast<const __nv_bfloat16*>(L.w_g);
  p.b_g = L.b_g; p.alpha = L.alpha;
  p.Q = pl.Q; p.P = pl.P; p.tiles = pl.tiles; p.nchunks = pl.nchunks; p.units = pl.units;
  p.max_tiles = pl.max_tiles; p.max_parts = pl.max_parts; p.ng = pl.ng;
  char* base = reinterpret_cast<char*>(ws);
  p.ws_sync = reinterpret_cast<unsigned*>(base + pl.off_sync);
  p.ws_tile_cnt = reinterpret_cast<unsigned*>(base + pl.off_cnt);
  p.ws_prod = reinterpret_cast<float*>(base + pl.off_prod);
  p.ws_T = reinterpret_cast<float*>(base + pl.off_T);
  p.ws_part = reinterpret_cast<float*>(base + pl.off_part);

  // Plans of other shapes may have changed this kernel's shared-memory limit
  // since this plan's grid was validated: restore the validated setting.
  if (int rc = cuda_check(cudaFuncSetAttribute(pl.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem),
                          "decode: smem attribute")) return rc;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(pl.Q + pl.P);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;        // every block resident: the T wait always ends
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_check(cudaLaunchKernelEx(&cfg, pl.fn, p), "decode launch");
}

// ---------------------------------------------------------------------------
// Decode without a caller workspace.  Some callers cannot allocate device
// memory when they call the layer: plugins hosted by a framework that owns the
// device allocator, runtimes that plan every buffer before serving starts and
// forbid allocation afterwards, and code on latency-critical paths where an
// allocation could synchronise the device.  For them the decode scratch lives
// in one fixed array in this module (kNoallocScratchBytes, held by every GPU
// that loads the library until the process exits).
constexpr size_t kNoallocScratchBytes = size_t(8) << 20;   // 8 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

namespace {
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {};      // device address of the scratch array, per device

// Once per device, with that device current: the array's device address (the
// symbol itself is only a host-side stand-in) and one zero fill.
int noalloc_scratch(void** out) {
  int dev = 0;
  if (int rc = cuda_check(cudaGetDevice(&dev), "cudaGetDevice")) return rc;
  if (dev < 0 || dev >= 64) return fail(SPEAR_ERR_UNSUPPORTED, "device index %d", dev);
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* ptr = nullptr;
    if (int rc = cuda_check(cudaGetSymbolAddress((void**)&ptr, g_noalloc_scratch), "decode scratch address"))
      return rc;
    if (int rc = cuda_check(cudaMemset(ptr, 0, kNoallocScratchBytes), "decode scratch zero fill")) return rc;
    g_noalloc_ptr[dev] = ptr;
  }
  *out = g_noalloc_ptr[dev];
  return SPEAR_OK;
}
}  // namespace

int launch_decode_noalloc(const spear_w4_layer& L, const uint16_t* x, int M, void* y, int out_f32,
                          cudaStream_t st) {
  Plan pl;
  if (int rc = get_plan(L, M, &pl)) return rc;
  if (pl.total > kNoallocScratchBytes)
    return fail(SPEAR_ERR_UNSUPPORTED,
                "decode_noalloc: N=%d K=%d M=%d needs %zu B of scratch; the built-in scratch holds %zu B",
                L.N, L.K, M, pl.total, kNoallocScratchBytes);
  void* ws = nullptr;
  if (int rc = noalloc_scratch(&ws)) return rc;
  // the synchronisation words and tile counters must start at zero
  if (int rc = cuda_check(cudaMemsetAsync(ws, 0, pl.off_prod, st), "decode scratch clear")) return rc;
  return launch_decode(L, x, M, y, out_f32, ws, kNoallocScratchBytes, st);
}

int read_and_clear_status_decode(unsigned* out, cudaStream_t st) {
  void* addr = nullptr;
  if (int rc = cuda_check(cudaGetSymbolAddress(&addr, g_decode_status), "decode status address")) return rc;
  if (int rc = cuda_check(cudaMemcpyAsync(out, addr, sizeof(unsigned), cudaMemcpyDeviceToHost, st), "read decode status")) return rc;
  if (int rc = cuda_check(cudaStreamSynchronize(st), "read decode status")) return rc;
  return cuda_check(cudaMemsetAsync(addr, 0, sizeof(unsigned), st), "clear decode status");
}

}  // namespace spear
