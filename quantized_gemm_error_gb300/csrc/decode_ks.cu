// decode_ks.cu -- decode kernel of the gated W4 + low-rank compensated linear
// for 1..32 tokens: one launch per layer, the compensator inside it (SPEAR
// explainer, Technical Summary 2.2 A: in the memory-bound decode phase the
// error compensator is fused into the low-bit GEMM, a single kernel).
//
//   y[m][n] = sum_k (u[n][k] - z[n][g]) s[n][g] x[m][k]  +  sum_j B[n][j] T[m][j]
//   T[m][j] = alpha g_m (A x_m)[j],   g_m = sigmoid(w_g . x_m + b_g)
//   (vector gate: T[m][j] = alpha gamma_j(t_m) t_m[j], t_m = A x_m)
//
// Work split.  Thread-block clusters of C CTAs; cluster g owns a range of
// 8-row weight tiles (N split G ways), CTA rank j of it a range of 128-k
// chunks (K split C ways).  Each CTA streams its rows x chunks of int4 codes
// once, by TMA, through a ring of stages; a stage is one chunk of a group of
// its rows together with the matching chunk of the tokens (and, in the first
// row group, of [A; w_g]).  The partial sums of the C CTAs meet in distributed
// shared memory: every CTA finishes 1/C of each row group's tiles.  The
// down-projection P = [A; w_g] x needs all of K, so every cluster computes it
// for itself (its CTAs over their K slices, the C partials summed by each
// CTA); nothing travels through global memory but the operands and y, and no
// CTA waits for another cluster.
//
// CTA roles (320 threads):
//   warps 0-7  consumers: for each stage and each of their tiles, turn the
//              int4 codes into exact integers (u - z) in bf16 registers and
//              multiply them by the tokens with mma.sync m16n8k16 (tokens as
//              the 16-row A operand, 8 weight rows as the B operand, fp32
//              accumulate); the group scale multiplies each 128-k partial in
//              fp32.  The bf16 products are exact, so the tokens keep their
//              full bf16 range.  Compensator tiles multiply bf16 rows of A.
//   warp 8     rearranges each stage's token chunk in place into the MMA's
//              A-fragment order (one shared-memory load per fragment later);
//   warp 9     one thread issues the TMA loads (weights first: they do not
//              depend on the kernel before this one).
//
// Within every 8-k group both operands take k in the order 0,4,1,5,2,6,3,7:
// the order in which two nibbles per mask come out of a 32-bit word of codes.
// Every 16-k MMA still sums the same products as the natural order.
//
// HBM traffic per call: N K / 2 (codes) + N K/G 2 (scales) + zeros + the
// tokens, (r+1) K 2 (A, w_g), N r 2 (B) and M N 2 (y); A and x are read once
// per cluster from L2.
#include <cuda.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"
#include "tmap.h"

namespace spear {
namespace {

__device__ unsigned g_dks_status;

using namespace sm100;

constexpr int kCW = 8;                       // consumer warps
constexpr int kXWarp = kCW;                  // token-fragment warp
constexpr int kTmaWarp = kCW + 1;            // TMA warp
constexpr int kThreads = (kCW + 2) * 32;     // 320
constexpr int kConsumers = kCW * 32;
constexpr int kChunkK = 128;
constexpr int kMaxC = 8;
constexpr int kMaxStages = 4;
constexpr int kMaxBoxRows = 256;             // TMA box limit; each TMA instruction costs ~55 ns to issue
constexpr int kMaxCompTilesPerWarp = 2;       // (rank + 1) / 8 rounded up <= 9 tiles over 8 warps
constexpr uint64_t kWaitNs = 2000ull * 1000 * 1000;  // 2 s: far beyond any legitimate wait

struct KsParams {
  int N, K, M, sym, ng;
  int C, G;                   // CTAs per cluster (K slices), clusters (row blocks)
  int tiles, nch;             // N / 8, K / 128
  int tcs;                    // compensator tiles of the row split (rank > 0), whether or not it runs
  int r;                      // rank when the compensator runs, else 0
  int rg_max;                 // most weight tiles one row group holds (the compensator tiles come on top, in the first)
  int S;                      // ring stages
  int box_rows;               // weight rows per TMA box (a multiple of 8, <= 256)
  uint32_t stage_bytes, off_x, off_a, off_cf;   // stage: codes at 0, tokens at off_x, [A; w_g] at off_a,
                                               // per-row coefficients at off_cf
  uint32_t off_sc, off_z, off_B, off_y, off_p, off_yr, off_t, off_g, off_h;
  int sc_cols, z_cols;        // staged scale columns / zero-point bytes per row
  int meta_async;             // scales and zero points may be copied with 4-byte cp.async
  const __half* scales;
  const uint8_t* zeros;
  void* y;
  int out_f32;
  const __nv_bfloat16* B;
  const __nv_bfloat16* w_g;
  float b_g, alpha;
  int gh;                     // vector-gate hidden width (0: the scalar gate)
  const float *gw1, *gc1, *gw2, *gc2;
  uint64_t wait_ns;           // limit of every bounded wait
};

struct Geo {
  int j, g;                   // cluster rank (K slice), cluster index (row block)
  int t0, T;                  // first tile, tile count
  int c0, nc;                 // first chunk, chunk count
  int nrg;                    // row groups
};

__device__ __forceinline__ Geo geometry(const KsParams& p) {
  Geo q;
  q.j = (int)cluster_ctarank();
  q.g = (int)blockIdx.x / p.C;
  q.t0 = q.g * p.tiles / p.G;                    // (products stay far below 2^31: tiles <= 2^24)
  q.T = (q.g + 1) * p.tiles / p.G - q.t0;
  q.c0 = q.j * p.nch / p.C;
  q.nc = (q.j + 1) * p.nch / p.C - q.c0;
  q.nrg = max(1, (q.T + p.rg_max - 1) / p.rg_max);
  return q;
}

// Weight tiles [s, s + n) of row group i (an even split; the compensator
// tiles join the first group).
__device__ __forceinline__ void rg_range(const KsParams& p, const Geo& q, int i, int& s, int& n) {
  s = i * q.T / q.nrg;
  n = (i + 1) * q.T / q.nrg - s;
}

__device__ __forceinline__ void give_up(int* abort_flag) {
  record_status(&g_dks_status, DEV_ERR_TIMEOUT);
  atomicExch(abort_flag, 1);
}

template <int MT, bool PERCH, bool COMP, int TPW>
__global__ void __launch_bounds__(kThreads, MT == 1 ? 2 : 1)
decode_ks_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                 const __grid_constant__ CUtensorMap tm_a, const KsParams p) {
  constexpr int MP = 16 * MT;                          // token rows of a stage
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_align_up(smem_raw, 1024);
  __shared__ __align__(8) uint64_t full[kMaxStages], empty[kMaxStages], xready[kMaxStages];
  __shared__ __align__(8) uint64_t ready_bar, done_bar, meta_bar;
  __shared__ int s_abort;

  pdl_launch_dependents();                             // let the next kernel on the stream start queueing
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const Geo q = geometry(p);
  const int nst = q.nrg * q.nc;                        // stages of this CTA
  const int n0 = 8 * q.t0;                             // first weight row of the CTA
  const int rows_c = 8 * p.tcs;
  __half* const sc_s = reinterpret_cast<__half*>(smem + p.off_sc);   // [8 T][sc_cols] the CTA's scales
  uint8_t* const z_s = smem + p.off_z;                                // [8 T][z_cols] its zero-point bytes
  const int sc0 = q.c0 & ~1;                           // first staged scale column
  const int zb0 = PERCH ? 0 : (q.c0 / 2) & ~3;         // first staged zero-point byte
  const int zrow = (p.ng + 1) / 2;

  if (threadIdx.x == 0) {
    for (int i = 0; i < p.S; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), kCW);
      mbar_init(smem_u32(&xready[i]), 1);
    }
    mbar_init(smem_u32(&ready_bar), p.C);
    mbar_init(smem_u32(&done_bar), p.C);
    mbar_init(smem_u32(&meta_bar), 1);
    s_abort = 0;
    fence_mbar_init();
  }
  // compensator rows the TMA never writes (padding past rank + 1, and the
  // gate row when the vector gate leaves w_g out) stay zero in every stage
  if (COMP && warp < kCW) {
    const int first = p.w_g && p.gh == 0 ? p.r + 1 : p.r;
    const int words = (rows_c - first) * (kChunkK * 2 / 16);
    for (int e = threadIdx.x; e < p.S * words; e += kConsumers) {
      const int st = e / words, w = e % words;
      *reinterpret_cast<uint4*>(smem + st * p.stage_bytes + p.off_a + first * kChunkK * 2 + w * 16) =
          make_uint4(0, 0, 0, 0);
    }
  }
  __syncthreads();
  // Cluster barrier, split: every thread arrives now, and waits only before
  // its first access to another CTA (the row-group epilogue) or before it
  // exits, so the barrier's latency hides under the weight stream.
  cluster_arrive_relaxed();

  auto slot_base = [&](int s) { return smem + (s % p.S) * p.stage_bytes; };
  auto nbox = [&](int n) { return (8 * n + p.box_rows - 1) / p.box_rows; };
  auto stage_tx = [&](int rg, int n) -> uint32_t {
    uint32_t b = (uint32_t)nbox(n) * p.box_rows * (kChunkK / 2) + MP * kChunkK * 2;
    if (COMP && rg == 0) b += p.r * kChunkK * 2 + (p.w_g && p.gh == 0 ? kChunkK * 2 : 0);
    return b;
  };

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------- TMA
    if (lane == 0) {
      int issued = 0;
      bool ok = true;
      prefetch_tmap(&tm_w);
      prefetch_tmap(&tm_x);
      if (COMP) prefetch_tmap(&tm_a);
      auto issue_w = [&](int s) {
        const int rg = s / q.nc, ch = s % q.nc;
        int rs, rn;
        rg_range(p, q, rg, rs, rn);
        const uint32_t bar = smem_u32(&full[s % p.S]);
        uint8_t* base = slot_base(s);
        for (int b = 0; b < nbox(rn); ++b)
          tma_load_2d(smem_u32(base + b * p.box_rows * (kChunkK / 2)), &tm_w, (q.c0 + ch) * (kChunkK / 2),
                      n0 + 8 * rs + p.box_rows * b, bar);
      };
      auto issue_rest = [&](int s) {
        const int rg = s / q.nc, ch = s % q.nc;
        const uint32_t bar = smem_u32(&full[s % p.S]);
        uint8_t* base = slot_base(s);
        tma_load_2d(smem_u32(base + p.off_x), &tm_x, (q.c0 + ch) * kChunkK, 0, bar);
        if (COMP && rg == 0) {
          tma_load_2d(smem_u32(base + p.off_a), &tm_a, (q.c0 + ch) * kChunkK, 0, bar);
          if (p.w_g && p.gh == 0)
            bulk_load_1d(smem_u32(base + p.off_a + p.r * kChunkK * 2), p.w_g + (size_t)(q.c0 + ch) * kChunkK,
                         kChunkK * 2, bar);
        }
      };
      const int pre = min(p.S, nst);
      // the first stages' codes read only the layer's weights: issued before
      // waiting for the kernel ahead (overlapped launches)
      for (int s = 0; s < pre; ++s) {
        int rs, rn;
        rg_range(p, q, s / q.nc, rs, rn);
        mbar_arrive_expect_tx(smem_u32(&full[s]), stage_tx(s / q.nc, rn));
        issue_w(s);
      }
      pdl_wait();                                      // tokens may come from the kernel ahead
      for (int s = 0; s < pre; ++s) issue_rest(s);
      issued = pre;
      for (int s = pre; s < nst && ok; ++s) {
        ok = mbar_wait(smem_u32(&empty[s % p.S]), ((s / p.S) & 1) ^ 1, p.wait_ns) && !s_abort;
        if (!ok) break;
        int rs, rn;
        rg_range(p, q, s / q.nc, rs, rn);
        mbar_arrive_expect_tx(smem_u32(&full[s % p.S]), stage_tx(s / q.nc, rn));
        issue_w(s);
        issue_rest(s);
        ++issued;
      }
      if (!ok) {
        give_up(&s_abort);
        // never leave with copies in flight: wait (bounded) for every issued fill
        for (int s = max(0, issued - p.S); s < issued; ++s)
          mbar_wait(smem_u32(&full[s % p.S]), (s / p.S) & 1, p.wait_ns);
      }
    }
    __syncwarp();
    cluster_wait();
    return;
  }

  if (warp == kXWarp) {
    // ------------------------------------------------ per-stage preparation
    // (1) the token chunk -> A-fragment order, in place, and per-token sums;
    // (2) per row of the stage the coefficients (s, -(128 + z) s) that turn
    //     the MMA's sum_k (128 + u) x into s sum_k (u - z) x (s = 1 for
    //     per-channel layers, whose scale multiplies the final sum).
    bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&meta_bar), 0, p.wait_ns));
    for (int s = 0; s < nst && ok; ++s) {
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&full[s % p.S]), (s / p.S) & 1, p.wait_ns) && !s_abort);
      if (!ok) break;
      uint8_t* xs = slot_base(s) + p.off_x;
      uint4 v[MT][4][2];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          v[mt][w][0] = *reinterpret_cast<const uint4*>(xs + (16 * mt + g) * (kChunkK * 2) + 64 * c + 16 * w);
          v[mt][w][1] = *reinterpret_cast<const uint4*>(xs + (16 * mt + g + 8) * (kChunkK * 2) + 64 * c + 16 * w);
        }
      __syncwarp();
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint4 lo = v[mt][w][0], hi = v[mt][w][1];      // tokens g and g + 8, k 8w' .. 8w' + 7
          // fragment h = 0 takes k (0,4) and (1,5); h = 1 takes (2,6) and (3,7)
          const uint4 f0 = make_uint4(__byte_perm(lo.x, lo.z, 0x5410), __byte_perm(hi.x, hi.z, 0x5410),
                                      __byte_perm(lo.x, lo.z, 0x7632), __byte_perm(hi.x, hi.z, 0x7632));
          const uint4 f1 = make_uint4(__byte_perm(lo.y, lo.w, 0x5410), __byte_perm(hi.y, hi.w, 0x5410),
                                      __byte_perm(lo.y, lo.w, 0x7632), __byte_perm(hi.y, hi.w, 0x7632));
          *reinterpret_cast<uint4*>(xs + ((mt * 4 + w) * 2 + 0) * 512 + lane * 16) = f0;
          *reinterpret_cast<uint4*>(xs + ((mt * 4 + w) * 2 + 1) * 512 + lane * 16) = f1;
        }
      // per-token sums of the chunk (fp32, fixed order: the lane's 32 k, then
      // the four lanes of a token row)
      float* xsum = reinterpret_cast<float*>(xs + MP * kChunkK * 2);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        float slo = 0.0f, shi = 0.0f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint32_t a[4] = {v[mt][w][0].x, v[mt][w][0].y, v[mt][w][0].z, v[mt][w][0].w};
          const uint32_t b[4] = {v[mt][w][1].x, v[mt][w][1].y, v[mt][w][1].z, v[mt][w][1].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            slo += bf16x2_lo(a[e]) + bf16x2_hi(a[e]);
            shi += bf16x2_lo(b[e]) + bf16x2_hi(b[e]);
          }
        }
        slo += __shfl_xor_sync(0xffffffffu, slo, 1);
        shi += __shfl_xor_sync(0xffffffffu, shi, 1);
        slo += __shfl_xor_sync(0xffffffffu, slo, 2);
        shi += __shfl_xor_sync(0xffffffffu, shi, 2);
        if (c == 0) {
          xsum[16 * mt + g] = slo;
          xsum[16 * mt + g + 8] = shi;
        }
      }
      fence_proxy_async_smem();                        // the next TMA fill of this slot comes after these writes
      {
        const int rg = s / q.nc, ch = s % q.nc, chg = q.c0 + ch;
        const int gi = PERCH ? 0 : chg;                // group of this chunk
        int rs, rn;
        rg_range(p, q, rg, rs, rn);
        float2* cf = reinterpret_cast<float2*>(slot_base(s) + p.off_cf);
        for (int e = lane; e < 8 * rn; e += 32) {
          const int row = 8 * rs + e;                  // row of the CTA
          const float sv = PERCH ? 1.0f : __half2float(sc_s[row * p.sc_cols + chg - sc0]);
          const int z = p.sym ? 8 : (z_s[row * p.z_cols + gi / 2 - zb0] >> (4 * (gi & 1))) & 15;
          cf[e] = make_float2(sv, -(float)(128 + z) * sv);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&xready[s % p.S]));
    }
    if (!ok) give_up(&s_abort);
    cluster_wait();
    return;
  }

  // ------------------------------------------------------------ consumers
  const int tid = threadIdx.x;                         // 0 .. kConsumers - 1
  __nv_bfloat16* B_s = reinterpret_cast<__nv_bfloat16*>(smem + p.off_B);
  float* ybuf = reinterpret_cast<float*>(smem + p.off_y);     // [rg tiles][MP][8] own partial
  float* pbuf = reinterpret_cast<float*>(smem + p.off_p);     // [tcs][MP][8] own partial of P
  float* yred = reinterpret_cast<float*>(smem + p.off_yr);    // [owned tiles][MP][8] cluster sums
  float* tfull = reinterpret_cast<float*>(smem + p.off_t);    // [MP][r + 1] t and the gate logit
  // T hi [MP][r/2], then lo [MP][r/2]: after the partial of P, which the
  // peers read until their done arrival
  uint32_t* thl = reinterpret_cast<uint32_t*>(smem + p.off_p + (size_t)p.tcs * 8 * MP * 8 * 4);
  float* gate_s = reinterpret_cast<float*>(smem + p.off_g);
  float* hid_s = reinterpret_cast<float*>(smem + p.off_h);

  // The CTA's scales and zero points (all its rows x its chunks), read only
  // from the layer's weights: before waiting for the kernel ahead.  4-byte
  // cp.async copies where the rows allow (an even number of groups per row,
  // zero-point rows a multiple of 4 bytes), else plain loads.
  {
    const int nrow = 8 * q.T;
    if (p.meta_async) {
      if (PERCH) {
        for (int e = tid; e < nrow / 2; e += kConsumers) cp_async4(sc_s + 2 * e, p.scales + (size_t)n0 + 2 * e);
      } else {
        const int pairs = p.sc_cols / 2;
        for (int e = tid; e < nrow * pairs; e += kConsumers) {
          const int row = e / pairs, col = sc0 + 2 * (e % pairs);
          if (col < p.ng) cp_async4(sc_s + row * p.sc_cols + (col - sc0), p.scales + (size_t)(n0 + row) * p.ng + col);
        }
      }
      if (!p.sym) {
        const int quads = p.z_cols / 4;
        for (int e = tid; e < nrow * quads; e += kConsumers) {
          const int row = e / quads, col = zb0 + 4 * (e % quads);
          if (col < zrow) cp_async4(z_s + row * p.z_cols + (col - zb0), p.zeros + (size_t)(n0 + row) * zrow + col);
        }
      }
    } else {
      const int cols = p.sc_cols;
      for (int e0 = tid; e0 < nrow * cols; e0 += 8 * kConsumers) {
        __half v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int e = e0 + u * kConsumers;
          const int row = e / cols, col = PERCH ? e % cols : sc0 + e % cols;
          v[u] = (e < nrow * cols && col < p.ng) ? p.scales[(size_t)(n0 + row) * p.ng + col] : __half();
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (e0 + u * kConsumers < nrow * cols) sc_s[e0 + u * kConsumers] = v[u];
      }
      if (!p.sym) {
        const int zc = p.z_cols;
        for (int e0 = tid; e0 < nrow * zc; e0 += 8 * kConsumers) {
          uint8_t v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int e = e0 + u * kConsumers;
            const int row = e / zc, col = zb0 + e % zc;
            v[u] = (e < nrow * zc && col < zrow) ? p.zeros[(size_t)(n0 + row) * zrow + col] : 0;
          }
#pragma unroll
          for (int u = 0; u < 8; ++u)
            if (e0 + u * kConsumers < nrow * zc) z_s[e0 + u * kConsumers] = v[u];
        }
      }
    }
    cp_async_commit();                                 // group: scales and zero points
  }
  if (COMP && p.gh > 0) stage_gate_weights_async(p.gw1, p.gw2, p.gc1, p.gc2, p.r, p.gh, gate_s, tid, kConsumers);
  else cp_async_commit();                              // (an empty group keeps the count)
  pdl_wait();                                          // y follows the kernel ahead

  bool ok = true;
  auto wait_local = [&](uint64_t* bar, uint32_t parity) {
    ok = __all_sync(0xffffffffu, ok && !s_abort && mbar_wait(smem_u32(bar), parity, p.wait_ns));
  };
  auto wait_cluster = [&](uint64_t* bar, uint32_t parity) {
    ok = __all_sync(0xffffffffu, ok && !s_abort && mbar_wait_cluster(smem_u32(bar), parity, p.wait_ns));
  };

  int stage = 0;
  bool cluster_ready = false;
  for (int rg = 0; rg < q.nrg; ++rg) {
    int rs, rn;
    rg_range(p, q, rg, rs, rn);
    const int o0 = q.j * rn / p.C, o1 = (q.j + 1) * rn / p.C;        // tiles finished here
    // peers have finished reading this CTA's partial of the previous row group
    if (rg > 0) wait_cluster(&done_bar, (rg - 1) & 1);
    // the factor-B rows of the tiles finished here (rows contiguous in B)
    if (COMP) {
      const int per = p.r / 8;                         // 16-byte pieces per row
      const int nb = 8 * (o1 - o0) * per;
      for (int e = tid; e < nb; e += kConsumers)
        cp_async16(B_s + (size_t)e * 8, p.B + (size_t)(n0 + 8 * (rs + o0)) * p.r + (size_t)e * 8);
    }
    cp_async_commit();                                 // group: this row group's B rows
    if (rg == 0) {
      cp_async_wait<2>();                              // the scales and zero points
      named_sync(1, kConsumers);
      if (tid == 0) mbar_arrive(smem_u32(&meta_bar));  // the stage preparation may use them
    }

    for (int ch = 0; ch < q.nc; ++ch, ++stage) {
      const int slot = stage % p.S;
      wait_local(&full[slot], (stage / p.S) & 1);
      wait_local(&xready[slot], (stage / p.S) & 1);
      if (ok) {
        const uint8_t* base = slot_base(stage);
        const float* xsum = reinterpret_cast<const float*>(base + p.off_x + MP * kChunkK * 2);
        const float4* cf = reinterpret_cast<const float4*>(base + p.off_cf);   // (s, z s) of rows 2i, 2i + 1
        const bool first = ch == 0;                    // the partial starts here
        if (rn > 0) {
          // Weight tiles of this warp: t = warp + 8 i, i < TPW.  No branch per
          // tile: indices past the row group repeat its last tile and their
          // results are dropped.  The codes enter the MMA as 128 + u (exact in
          // bf16, no per-word subtraction); s sum_k (128 + u) x - (128 + z) s
          // sum_k x follows per chunk.  The four 32-k word steps each feed
          // every tile, so the tiles' MMA chains are independent.
          uint4 wv[TPW];
#pragma unroll
          for (int i = 0; i < TPW; ++i) {
            const int t = min(warp + kCW * i, rn - 1);
            wv[i] = *reinterpret_cast<const uint4*>(base + t * 512 + g * 64 + c * 16);
          }
          float X[MT][2];
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            X[mt][0] = xsum[16 * mt + g];
            X[mt][1] = xsum[16 * mt + g + 8];
          }
          float part[TPW][MT][4];
#pragma unroll
          for (int i = 0; i < TPW; ++i)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
              for (int e = 0; e < 4; ++e) part[i][mt][e] = 0.0f;
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            uint4 xa[MT][2];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
              for (int h = 0; h < 2; ++h)
                xa[mt][h] = *reinterpret_cast<const uint4*>(base + p.off_x + ((mt * 4 + w) * 2 + h) * 512 + lane * 16);
#pragma unroll
            for (int i = 0; i < TPW; ++i) {
              const uint32_t word = w == 0 ? wv[i].x : w == 1 ? wv[i].y : w == 2 ? wv[i].z : wv[i].w;
              uint32_t o[4];
              nibbles_to_bf16x2_biased(word, o);       // 128 + u
#pragma unroll
              for (int mt = 0; mt < MT; ++mt) {
                mma_bf16_16816(part[i][mt], xa[mt][0].x, xa[mt][0].y, xa[mt][0].z, xa[mt][0].w, o[0], o[1]);
                mma_bf16_16816(part[i][mt], xa[mt][1].x, xa[mt][1].y, xa[mt][1].z, xa[mt][1].w, o[2], o[3]);
              }
            }
          }
          // partial += s part + (z s) sum x in the shared-memory partial
          // (each lane owns its C-fragment elements: tokens g, g + 8, rows
          // 2c, 2c + 1 of the tile)
#pragma unroll
          for (int i = 0; i < TPW; ++i) {
            const int t = warp + kCW * i;
            const int tc = min(t, rn - 1);
            const float4 k = cf[4 * tc + c];           // rows 8 tc + 2c and 8 tc + 2c + 1
            float* dst = ybuf + (size_t)tc * MP * 8;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              float2* d0 = reinterpret_cast<float2*>(dst + (16 * mt + g) * 8 + 2 * c);
              float2* d1 = reinterpret_cast<float2*>(dst + (16 * mt + g + 8) * 8 + 2 * c);
              const float2 a0 = first ? make_float2(0.0f, 0.0f) : *d0;
              const float2 a1 = first ? make_float2(0.0f, 0.0f) : *d1;
              const float2 r0 = make_float2(fmaf(k.x, part[i][mt][0], fmaf(k.y, X[mt][0], a0.x)),
                                            fmaf(k.z, part[i][mt][1], fmaf(k.w, X[mt][0], a0.y)));
              const float2 r1 = make_float2(fmaf(k.x, part[i][mt][2], fmaf(k.y, X[mt][1], a1.x)),
                                            fmaf(k.z, part[i][mt][3], fmaf(k.w, X[mt][1], a1.y)));
              if (t < rn) {
                *d0 = r0;
                *d1 = r1;
              }
            }
          }
        }
        if (COMP && rg == 0) {
          // compensator tiles: 8 rows of [A; w_g] in bf16, as they are
#pragma unroll
          for (int j = 0; j < kMaxCompTilesPerWarp; ++j) {
            const int ct = warp + kCW * j;
            if (ct < p.tcs) {
              float cp[MT][4];
#pragma unroll
              for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) cp[mt][e] = 0.0f;
              const uint8_t* arow = base + p.off_a + (8 * ct + g) * (kChunkK * 2) + 64 * c;
#pragma unroll
              for (int w = 0; w < 4; ++w) {
                const uint4 av = *reinterpret_cast<const uint4*>(arow + 16 * w);
                const uint32_t b0 = __byte_perm(av.x, av.z, 0x5410), b1 = __byte_perm(av.x, av.z, 0x7632);
                const uint32_t b2 = __byte_perm(av.y, av.w, 0x5410), b3 = __byte_perm(av.y, av.w, 0x7632);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                  const uint4 x0 = *reinterpret_cast<const uint4*>(base + p.off_x + ((mt * 4 + w) * 2 + 0) * 512 + lane * 16);
                  const uint4 x1 = *reinterpret_cast<const uint4*>(base + p.off_x + ((mt * 4 + w) * 2 + 1) * 512 + lane * 16);
                  mma_bf16_16816(cp[mt], x0.x, x0.y, x0.z, x0.w, b0, b1);
                  mma_bf16_16816(cp[mt], x1.x, x1.y, x1.z, x1.w, b2, b3);
                }
              }
              float* dst = pbuf + (size_t)ct * MP * 8;
#pragma unroll
              for (int mt = 0; mt < MT; ++mt) {
                float2* d0 = reinterpret_cast<float2*>(dst + (16 * mt + g) * 8 + 2 * c);
                float2* d1 = reinterpret_cast<float2*>(dst + (16 * mt + g + 8) * 8 + 2 * c);
                const float2 a0 = first ? make_float2(0.0f, 0.0f) : *d0;
                const float2 a1 = first ? make_float2(0.0f, 0.0f) : *d1;
                *d0 = make_float2(a0.x + cp[mt][0], a0.y + cp[mt][1]);
                *d1 = make_float2(a1.x + cp[mt][2], a1.y + cp[mt][3]);
              }
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[slot]));
    }

    // ------------------------------------------ row-group epilogue (cluster)
    named_sync(1, kConsumers);
    if (!cluster_ready) {                              // every peer's barriers are initialised
      cluster_wait();
      cluster_ready = true;
    }
    // one lane per peer: the arrives (release, cluster scope) go out together
    if (warp == 0 && lane < p.C && ok && !s_abort) mbar_arrive_remote(dsmem_addr(smem_u32(&ready_bar), (uint32_t)lane));
    wait_cluster(&ready_bar, rg & 1);
    // every CTA's partials are in place: sum P (first row group) and this
    // CTA's tiles over the cluster, in rank order, all loads in flight
    if (ok) {
      const int pu = (COMP && rg == 0) ? p.tcs * MP * 2 : 0;          // float4 units of P
      const int yu = (o1 - o0) * MP * 2;                               // float4 units of owned rows
      const uint32_t pb = smem_u32(pbuf), yb = smem_u32(ybuf) + (uint32_t)o0 * MP * 8 * 4;
      for (int e = tid; e < pu + yu; e += kConsumers) {
        const uint32_t la = e < pu ? pb + (uint32_t)e * 16 : yb + (uint32_t)(e - pu) * 16;
        // the peers' partials in rank order, four loads in flight at a time
        float4 sum = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
        for (int q0 = 0; q0 < kMaxC; q0 += 4) {
          float4 v[4];
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (q0 + u < p.C) v[u] = dsmem_ld_f32x4(dsmem_addr(la, (uint32_t)(q0 + u)));
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (q0 + u < p.C) { sum.x += v[u].x; sum.y += v[u].y; sum.z += v[u].z; sum.w += v[u].w; }
        }
        if (e < pu) {
          // P element units: compensator tile ct, token m, rows 4 h .. 4 h + 3
          const int ct = e / (MP * 2), m = (e / 2) % MP, h = e & 1;
          const float vv[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int row = 8 * ct + 4 * h + u;          // row of [A; w_g]
            if (row <= p.r) tfull[m * (p.r + 1) + row] = vv[u];
          }
        } else {
          reinterpret_cast<float4*>(yred)[e - pu] = sum;
        }
      }
    }
    named_sync(1, kConsumers);
    // this CTA's reads of the peers' partials are done
    if (warp == 0 && lane < p.C && ok && !s_abort) mbar_arrive_remote(dsmem_addr(smem_u32(&done_bar), (uint32_t)lane));

    if (COMP && rg == 0 && ok) {
      // T = alpha g t as bf16 hi + lo (hi + lo = T to ~2^-16 relative)
      const int rp = p.r + 1, hr = p.r / 2;
      uint32_t* th = thl;
      uint32_t* tl = thl + MP * hr;
      if (p.gh > 0) {
        cp_async_wait<1>();                            // the staged gate weights (the B rows may still land)
        named_sync(1, kConsumers);
        // vector gate over all tokens: t [MP][r] packed at stride r
        float* ts = tfull;
        for (int e = tid; e < MP * p.r; e += kConsumers) {
          const int m = e / p.r, jj = e % p.r;
          hid_s[e] = ts[m * rp + jj];                  // repack t at stride r (hid_s as scratch)
        }
        named_sync(1, kConsumers);
        for (int e = tid; e < MP * p.r; e += kConsumers) ts[e] = hid_s[e];
        named_sync(1, kConsumers);
        const GateSmem gt(gate_s, p.r, p.gh);
        vector_gate_hidden_rows(ts, MP, gt, hid_s, tid, kConsumers);
        named_sync(1, kConsumers);
        vector_gate_apply_rows(ts, MP, gt, hid_s, tid, kConsumers);
        named_sync(1, kConsumers);
        for (int e = tid; e < MP * hr; e += kConsumers) {
          const int m = e / hr, jj = 2 * (e % hr);
          const bool on = m < p.M;
          const float ta = on ? p.alpha * ts[m * p.r + jj] : 0.0f, tb = on ? p.alpha * ts[m * p.r + jj + 1] : 0.0f;
          const float ha = __bfloat162float(__float2bfloat16_rn(ta)), hb = __bfloat162float(__float2bfloat16_rn(tb));
          th[e] = pack_bf16x2(ha, hb);
          tl[e] = pack_bf16x2(ta - ha, tb - hb);
        }
      } else {
        for (int e = tid; e < MP * hr; e += kConsumers) {
          const int m = e / hr, jj = 2 * (e % hr);
          const float gm = m < p.M ? p.alpha / (1.0f + expf(-(tfull[m * rp + p.r] + p.b_g))) : 0.0f;
          const float ta = gm * tfull[m * rp + jj], tb = gm * tfull[m * rp + jj + 1];
          const float ha = __bfloat162float(__float2bfloat16_rn(ta)), hb = __bfloat162float(__float2bfloat16_rn(tb));
          th[e] = pack_bf16x2(ha, hb);
          tl[e] = pack_bf16x2(ta - ha, tb - hb);
        }
      }
    }
    cp_async_wait<0>();                                // the factor-B rows
    named_sync(1, kConsumers);

    // y for the tiles finished here: (tile, token tile) items over the warps
    if (ok) {
      const int hr = p.r / 2;
      const uint32_t* th = thl;
      const uint32_t* tl = thl + MP * hr;
      for (int item = warp; item < (o1 - o0) * MT; item += kCW) {
        const int ot = item / MT, mt = item % MT;
        const float* yr = yred + (size_t)ot * MP * 8;
        float d[4];
        const float2 lo = *reinterpret_cast<const float2*>(yr + (16 * mt + g) * 8 + 2 * c);
        const float2 hi = *reinterpret_cast<const float2*>(yr + (16 * mt + g + 8) * 8 + 2 * c);
        d[0] = lo.x; d[1] = lo.y; d[2] = hi.x; d[3] = hi.y;
        const int row0 = 8 * (rs + o0 + ot) + 2 * c;   // row of the CTA (d[0], d[2]: row0; d[1], d[3]: row0 + 1)
        if (PERCH) {
          const int rr = 8 * (rs + o0 + ot) + 2 * c;   // row of the CTA
          const float s0 = __half2float(sc_s[rr * p.sc_cols]), s1 = __half2float(sc_s[(rr + 1) * p.sc_cols]);
          d[0] *= s0; d[2] *= s0; d[1] *= s1; d[3] *= s1;
        }
        if (COMP) {
          const uint32_t* brow = reinterpret_cast<const uint32_t*>(B_s + (size_t)(8 * ot + g) * p.r);
          for (int j0 = 0; j0 < p.r; j0 += 16) {
            const uint32_t b0 = brow[j0 / 2 + c], b1 = brow[j0 / 2 + c + 4];
            const int ta = (16 * mt + g) * hr + j0 / 2, tb = (16 * mt + g + 8) * hr + j0 / 2;
            mma_bf16_16816(d, th[ta + c], th[tb + c], th[ta + c + 4], th[tb + c + 4], b0, b1);
            mma_bf16_16816(d, tl[ta + c], tl[tb + c], tl[ta + c + 4], tl[tb + c + 4], b0, b1);
          }
        }
        const int m0 = 16 * mt + g, m1 = m0 + 8;
        const size_t n = (size_t)n0 + row0;
        if (p.out_f32) {
          float* yf = reinterpret_cast<float*>(p.y);
          if (m0 < p.M) *reinterpret_cast<float2*>(yf + (size_t)m0 * p.N + n) = make_float2(d[0], d[1]);
          if (m1 < p.M) *reinterpret_cast<float2*>(yf + (size_t)m1 * p.N + n) = make_float2(d[2], d[3]);
        } else {
          __nv_bfloat16* yb = reinterpret_cast<__nv_bfloat16*>(p.y);
          if (m0 < p.M) *reinterpret_cast<uint32_t*>(yb + (size_t)m0 * p.N + n) = pack_bf16x2(d[0], d[1]);
          if (m1 < p.M) *reinterpret_cast<uint32_t*>(yb + (size_t)m1 * p.N + n) = pack_bf16x2(d[2], d[3]);
        }
      }
    }
    named_sync(1, kConsumers);                         // staged scales / B rows are reused by the next row group
  }
  // peers are done reading this CTA's shared memory (and arriving on its
  // barriers) before it exits: waited for even after a failure, bounded
  if (!mbar_wait_cluster(smem_u32(&done_bar), (q.nrg - 1) & 1, p.wait_ns)) ok = false;
  if (!ok) give_up(&s_abort);
}

using KsKernel = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, KsParams);

constexpr int tpw_for(int MT) { return MT == 1 ? 5 : 4; }    // tiles per consumer warp in a row group

template <int MT>
KsKernel pick_mt(bool perch, bool comp) {
  constexpr int T = tpw_for(MT);
  if (perch) return comp ? decode_ks_kernel<MT, true, true, T> : decode_ks_kernel<MT, true, false, T>;
  return comp ? decode_ks_kernel<MT, false, true, T> : decode_ks_kernel<MT, false, false, T>;
}

KsKernel pick_ks(int MT, bool perch, bool comp) { return MT == 1 ? pick_mt<1>(perch, comp) : pick_mt<2>(perch, comp); }

// ---------------------------------------------------------------- plan --
struct KsPlan {
  int device, N, K, G, rank, comp, MT, gh, sym;   // key
  int C, Gc, tiles, nch, tcs, rg_max, S, box_rows, meta_async;
  size_t smem;
  uint32_t stage_bytes, off_x, off_a, off_cf, off_sc, off_z, off_B, off_y, off_p, off_yr, off_t, off_g, off_h;
  int sc_cols, z_cols;
  KsKernel fn;
};

size_t up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Shared-memory layout for `rg_max` tiles per row group, S stages and the
// scales / zero points of `meta_rows` rows.
size_t layout(KsPlan* c, int rg_max, int S, int MP, int rank, int ncs_max, int nzs_max, int meta_rows) {
  const int rows_c = 8 * c->tcs;
  const int rows = 8 * rg_max;
  const int nb = (rows + kMaxBoxRows - 1) / kMaxBoxRows;
  c->box_rows = 8 * ((rows / 8 + nb - 1) / nb);
  size_t st = (size_t)nb * c->box_rows * (kChunkK / 2);
  c->off_x = (uint32_t)st;
  // token chunk (then its fragments) and token sums; every TMA destination
  // (codes at 0, tokens at off_x, [A; w_g] at off_a) 128-byte aligned
  st += (size_t)MP * kChunkK * 2 + up((size_t)MP * 4, 128);
  c->off_a = (uint32_t)st;
  st += (size_t)rows_c * kChunkK * 2;
  c->off_cf = (uint32_t)st;                       // (s, -(128 + z) s) per row of the stage
  st += (size_t)rows * 8;
  c->stage_bytes = (uint32_t)up(st, 1024);
  if (c->off_x % 128 != 0 || c->off_a % 128 != 0) return (size_t)-1;   // never: TMA needs 128-byte destinations
  size_t off = (size_t)S * c->stage_bytes;
  c->off_sc = (uint32_t)off;                     // the CTA's scales and zero points
  off = up(off + (size_t)meta_rows * ncs_max * 2, 16);
  c->off_z = (uint32_t)off;
  off = up(off + (size_t)meta_rows * nzs_max, 16);
  const int own_tiles = (rg_max + c->C - 1) / c->C + 1;
  c->off_B = (uint32_t)off;
  off = up(off + (size_t)own_tiles * 8 * std::max(rank, 8) * 2, 16);
  c->off_y = (uint32_t)off;
  off = up(off + (size_t)rg_max * MP * 8 * 4, 16);
  c->off_p = (uint32_t)off;                       // P partial, then T hi/lo
  off = up(off + (size_t)rows_c * MP * 8 * 4 + (size_t)MP * rank * 4, 16);
  c->off_yr = (uint32_t)off;
  off = up(off + (size_t)own_tiles * MP * 8 * 4, 16);
  c->off_t = (uint32_t)off;                       // t = A x and the gate logit
  off = up(off + (size_t)MP * (rank + 1) * 4, 16);
  c->off_g = (uint32_t)off;
  off = up(off + (c->gh > 0 ? (size_t)gate_smem_floats(rank, c->gh) * 4 : 0), 16);
  c->off_h = (uint32_t)off;                       // vector gate scratch: t repacked, hidden units
  off = up(off + (c->gh > 0 ? (size_t)MP * std::max(rank, gate_hid_stride(32)) * 4 : 0), 16);
  return off + 1024;                             // alignment slack of the dynamic base
}

int env_int(const char* name, int dflt) {
  const char* v = std::getenv(name);
  return (v && v[0]) ? std::atoi(v) : dflt;
}

int build_ks_plan(const spear_w4_layer& L, int MT, bool comp, const DeviceInfo& di, KsPlan* pl) {
  const bool perch = L.group_size == L.K;
  pl->MT = MT;
  pl->fn = pick_ks(MT, perch, comp);
  pl->tiles = L.N / 8;
  pl->nch = L.K / kChunkK;
  pl->tcs = L.rank > 0 ? (L.rank + 1 + 7) / 8 : 0;       // from the rank: the split does not depend on comp
  int C = env_int("SPEAR_KS_CLUSTER", 8);
  C = std::max(1, std::min(C, kMaxC));
  while (C > 1 && pl->nch < C) C /= 2;
  pl->C = C;
  const int MP = 16 * MT;

  // all of the shared memory a CTA may take (the kernel's static arrays aside)
  cudaFuncAttributes fa{};
  if (cudaFuncGetAttributes(&fa, pl->fn) != cudaSuccess) return fail(SPEAR_ERR_CUDA, "decode: cudaFuncGetAttributes failed");
  const size_t optin = di.smem_optin > fa.sharedSizeBytes ? di.smem_optin - fa.sharedSizeBytes : 0;
  if (int rc = ensure_smem_limit(reinterpret_cast<const void*>(pl->fn), optin)) return rc;
  cudaLaunchConfig_t cfg{};
  cfg.blockDim = dim3(kThreads);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // clusters: as many as fit with one CTA per SM (the SMs' other halves stay
  // free for the next kernel of an overlapped chain)
  cfg.gridDim = dim3(C);
  cfg.dynamicSmemBytes = optin;
  int max_clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&max_clusters, pl->fn, &cfg) != cudaSuccess || max_clusters < 1) {
    cudaGetLastError();
    return fail(SPEAR_ERR_UNSUPPORTED, "decode: no cluster of %d CTAs fits", C);
  }
  int Gc = env_int("SPEAR_KS_CLUSTERS", max_clusters);
  Gc = std::max(1, std::min(Gc, pl->tiles));
  pl->Gc = Gc;
  const int T_max = (pl->tiles + Gc - 1) / Gc;
  const int c_per = (pl->nch + C - 1) / C;
  const int ng = L.K / L.group_size;
  auto round_up = [](int v, int a) { return (v + a - 1) / a * a; };
  const int ncs_max = perch ? 1 : round_up(std::min(c_per + 2, ng + 1), 2);     // even: 4-byte copies
  const int nzs_max = (L.symmetric || perch) ? 4 : round_up(c_per / 2 + 8, 4);  // a multiple of 4 bytes
  const int zrow = (ng + 1) / 2;
  pl->meta_async = (perch || ng % 2 == 0) && (L.symmetric || (!perch && zrow % 4 == 0));

  const int rg_top = std::min(tpw_for(MT) * kCW, T_max);
  // two CTAs per SM when the layout allows it: the next kernel of an
  // overlapped chain then starts on the SMs while this one finishes
  int smem_sm = 0;
  cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, di.device);
  const size_t half = (size_t)smem_sm / 2 > 1024 + fa.sharedSizeBytes ? (size_t)smem_sm / 2 - 1024 - fa.sharedSizeBytes : 0;
  const size_t budgets[2] = {half, optin};
  bool found = false;
  for (size_t budget : budgets) {
    if (budget > optin) continue;
    for (int rg = rg_top; rg >= std::min(rg_top, 8) && !found; rg -= 2) {
      for (int S = kMaxStages; S >= 2 && !found; --S) {
        KsPlan c = *pl;
        const size_t sm = layout(&c, rg, S, MP, L.rank, ncs_max, nzs_max, 8 * T_max);
        if (sm <= budget) {
          c.rg_max = rg;
          c.S = S;
          c.smem = sm;
          c.sc_cols = ncs_max;
          c.z_cols = nzs_max;
          *pl = c;
          found = true;
        }
      }
    }
    if (found) break;
  }
  if (!found) return fail(SPEAR_ERR_UNSUPPORTED, "decode: no shared-memory layout for N=%d K=%d", L.N, L.K);
  return SPEAR_OK;
}

int get_ks_plan(const spear_w4_layer& L, int M, KsPlan* out) {
  DeviceInfo di;
  if (int rc = device_info(&di)) return rc;
  const int MT = M <= 16 ? 1 : 2;
  const int comp = (L.comp_enabled && L.rank > 0) ? 1 : 0;
  const int gh = comp ? L.gate_hidden : 0;
  static std::mutex mu;
  static std::vector<KsPlan> cache;
  std::lock_guard<std::mutex> lk(mu);
  for (const KsPlan& p : cache)
    if (p.device == di.device && p.N == L.N && p.K == L.K && p.G == L.group_size && p.rank == L.rank &&
        p.comp == comp && p.MT == MT && p.gh == gh && p.sym == L.symmetric) {
      *out = p;
      return SPEAR_OK;
    }
  KsPlan p{};
  p.gh = gh;
  if (int rc = build_ks_plan(L, MT, comp != 0, di, &p)) return rc;
  p.device = di.device; p.N = L.N; p.K = L.K; p.G = L.group_size; p.rank = L.rank; p.comp = comp; p.sym = L.symmetric;
  if (log_plans())
    fprintf(stderr, "[spear] decode ks plan N=%d K=%d G=%d rank=%d comp=%d MT=%d: C=%d clusters=%d rg_max=%d S=%d "
            "box_rows=%d stage=%u smem=%zu\n", L.N, L.K, L.group_size, L.rank, comp, MT, p.C, p.Gc, p.rg_max, p.S,
            p.box_rows, p.stage_bytes, p.smem);
  if (cache.size() > 4096) cache.clear();
  cache.push_back(p);
  *out = p;
  return SPEAR_OK;
}


}  // namespace

bool decode_ks_supports(const spear_w4_layer& L, int M) {
  if (M < 1 || M > 32) return false;
  if (!env_int("SPEAR_DECODE_KS", 0)) return false;     // opt-in while its tensor-core consumers are built
  KsPlan pl;
  char saved[512];
  snprintf(saved, sizeof(saved), "%s", spear_last_error());
  const int rc = get_ks_plan(L, M, &pl);
  if (rc != SPEAR_OK) set_last_error(saved);
  return rc == SPEAR_OK;
}


int launch_decode_ks(const spear_w4_layer& L, const uint16_t* x, int M, void* y, int out_f32, cudaStream_t st,
                     bool overlap) {
  KsPlan pl;
  if (int rc = get_ks_plan(L, M, &pl)) return rc;
  const int MP = 16 * pl.MT;
  const bool comp = pl.comp != 0;
  CUtensorMap tm_w, tm_x, tm_a;
  if (int rc = make_tmap(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, L.qweight, L.K / 2, L.N, kChunkK / 2, pl.box_rows,
                         CU_TENSOR_MAP_SWIZZLE_NONE)) return rc;
  if (int rc = make_tmap(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, L.K, M, kChunkK, MP,
                         CU_TENSOR_MAP_SWIZZLE_NONE)) return rc;
  if (comp) {
    if (int rc = make_tmap(&tm_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, L.A, L.K, L.rank, kChunkK, L.rank,
                           CU_TENSOR_MAP_SWIZZLE_NONE)) return rc;
  } else {
    tm_a = tm_x;                                   // never used
  }
  KsParams p{};
  p.N = L.N; p.K = L.K; p.M = M; p.sym = L.symmetric; p.ng = L.K / L.group_size;
  p.C = pl.C; p.G = pl.Gc; p.tiles = pl.tiles; p.nch = pl.nch; p.tcs = pl.tcs;
  p.r = comp ? L.rank : 0;
  p.rg_max = pl.rg_max; p.S = pl.S; p.box_rows = pl.box_rows;
  p.stage_bytes = pl.stage_bytes; p.off_x = pl.off_x; p.off_a = pl.off_a; p.off_cf = pl.off_cf;
  p.off_sc = pl.off_sc; p.off_z = pl.off_z; p.off_B = pl.off_B; p.off_y = pl.off_y; p.off_p = pl.off_p;
  p.off_yr = pl.off_yr; p.off_t = pl.off_t; p.off_g = pl.off_g; p.off_h = pl.off_h;
  p.sc_cols = pl.sc_cols; p.z_cols = pl.z_cols;
  p.meta_async = pl.meta_async;
  p.scales = reinterpret_cast<const __half*>(L.scales);
  p.zeros = L.zeros;
  p.y = y; p.out_f32 = out_f32;
  p.B = reinterpret_cast<const __nv_bfloat16*>(L.B);
  p.w_g = reinterpret_cast<const __nv_bfloat16*>(L.w_g);
  p.b_g = L.b_g; p.alpha = L.alpha;
  p.gh = comp ? L.gate_hidden : 0;
  p.gw1 = L.gate_w1; p.gc1 = L.gate_c1; p.gw2 = L.gate_w2; p.gc2 = L.gate_c2;
  p.wait_ns = wait_limit_ns(kWaitNs);

  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(pl.Gc * pl.C);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = pl.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 2 : 1;
  return cuda_check(cudaLaunchKernelEx(&cfg, pl.fn, tm_w, tm_x, tm_a, p), "decode launch");
}

int read_and_clear_status_decode_ks(unsigned* out, cudaStream_t st) {
  void* addr = nullptr;
  if (int rc = cuda_check(cudaGetSymbolAddress(&addr, g_dks_status), "decode status address")) return rc;
  if (int rc = cuda_check(cudaMemcpyAsync(out, addr, sizeof(unsigned), cudaMemcpyDeviceToHost, st),
                          "read decode status")) return rc;
  if (int rc = cuda_check(cudaStreamSynchronize(st), "read decode status")) return rc;
  return cuda_check(cudaMemsetAsync(addr, 0, sizeof(unsigned), st), "clear decode status");
}

}  // namespace spear
