// decode_tm.cu -- decode kernel of the gated W4 + low-rank compensated linear
// for 1..64 tokens on the 5th-generation tensor cores: one launch per layer,
// the compensator inside it (SPEAR explainer, Technical Summary 2.2 A: in the
// memory-bound decode phase the error compensator is fused into the low-bit
// GEMM, a single kernel).
//
//   y[m][n] = sum_k (u[n][k] - z[n][g]) s[n][g] x[m][k]  +  sum_j B[n][j] T[m][j]
//   T[m][j] = alpha g_m (A x_m)[j],   g_m = sigmoid(w_g . x_m + b_g)
//   (vector gate: T[m][j] = alpha gamma_j(t_m) t_m[j], t_m = A x_m)
//
// Work split.  Thread-block clusters of C CTAs; cluster g owns a range of
// 8-row weight tiles (N split G ways), CTA rank j of it a range of 128-k
// chunks (K split C ways).  Each CTA streams its rows x chunks of int4 codes
// once, by TMA, through a ring of stages; a stage is one chunk of a group of
// its rows (up to 3 slices of 128) with the matching chunk of the tokens (and,
// in the first row group, of [A; w_g]).  The C partial sums meet in
// distributed shared memory: every CTA finishes 1/C of each row group's rows.
// The down-projection P = [A; w_g] x needs all of K, so every cluster
// computes it for itself (its CTAs over their K slices, summed by every CTA);
// nothing crosses clusters, and no CTA waits for another cluster.
//
// The weights enter the tensor core from tensor memory.  A "pair" is one
// 128-row slice of a stage (or the stage's compensator rows):
//   * conversion warps (one per TMEM lane quarter and pair, two sets taking
//     alternate pairs) turn a row's 64 int4 bytes into 128 + u (exact in
//     bf16) and store them straight into one of four TMEM A buffers: the bf16
//     weights never pass through shared memory;
//   * one thread issues 8 tcgen05.mma (M = 128 rows, N = 16 / 32 / 64 tokens,
//     K = 16) per pair, the tokens (B operand) read from shared memory, into
//     a ring of per-chunk TMEM accumulators;
//   * reduction warps fold each chunk's accumulator into running sums held in
//     registers (one row and half the tokens per thread):
//       acc += s (sum_k (128 + u) x) - (128 + z) s (sum_k x)
//     with the group scale s and zero point z of the row and chunk.
//     Per-channel layers skip this: their MMAs accumulate over the whole K
//     slice in tensor memory, and the zero-point term and the scale are
//     applied once, in the epilogue.
// Conversion, MMA and reduction of consecutive pairs overlap: the rings hold
// four converted pairs and up to eight accumulators.  The reduction warps
// also run the row-group epilogue (cluster sum, gate, B T, store) while the
// conversion warps go on with the next row group.
// One warp turns each token chunk into the tensor core's K-major 128-byte
// swizzled layout (and per-token sums of the chunk); one issues the TMA
// loads; one allocates tensor memory and issues the MMAs.
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

__device__ unsigned g_dtm_status;

using namespace sm100;

constexpr int kSets = 3;                      // conversion sets: pair i goes to set i % kSets
constexpr int kCvt = 4 * kSets;               // conversion warps (one per TMEM lane quarter and set)
constexpr int kRed = 8;                       // reduction / epilogue warps (8 .. 15)
constexpr int kXWarp = kCvt + kRed;           // token-layout warp
constexpr int kTmaWarp = kXWarp + 1;          // TMA warp
constexpr int kMmaWarp = kXWarp + 2;          // TMEM allocation + MMA issue
constexpr int kThreads = (kXWarp + 3) * 32;   // 608
constexpr int kRedThreads = kRed * 32;
constexpr int kChunkK = 128;
constexpr int kMaxC = 8;
constexpr int kMaxStages = 4;
constexpr int kMaxBoxRows = 256;              // TMA box limit; each TMA instruction costs ~55 ns to issue
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitNs = 2000ull * 1000 * 1000;  // 2 s: far beyond any legitimate wait

// 128-row slices per row group: per-channel layers keep the slices' sums in
// tensor memory (3); per-group layers keep them in the reduction warps'
// registers (3 x 8, 2 x 16 or 1 x 32 floats a thread).
__host__ __device__ constexpr int tm_slices(int NT, bool perch) { return perch ? 3 : NT == 16 ? 3 : NT == 32 ? 2 : 1; }
// per-chunk accumulators of the ring (per-group layers): what is left of the
// 512 columns after the A buffers and P
__host__ __device__ constexpr int tm_dbufs(int NT) { return NT == 16 ? 7 : NT == 32 ? 7 : 3; }
// TMEM A buffers of 64 columns
__host__ __device__ constexpr int tm_abufs(int NT) { return NT == 16 ? 6 : 4; }

struct TmParams {
  int N, K, M, sym, ng;
  int C, G;                   // CTAs per cluster (K slices), clusters (row blocks)
  int tiles, nch;             // N / 8, K / 128
  int r;                      // rank when the compensator runs, else 0
  int rg_max;                 // most 8-row tiles one row group holds
  int S;                      // ring stages
  int box_rows;               // weight rows per TMA box (a multiple of 8, <= 256)
  // stage layout: codes at 0 (64-byte swizzle), raw tokens at off_x, the
  // tokens' MMA layout at off_xb (two 64-k panels, 128-byte swizzle), rows of
  // A at off_a (two panels, 128-byte swizzle), w_g at off_wg
  uint32_t stage_bytes, off_x, off_xb, off_a, off_wg;
  uint32_t off_sc, off_z, off_xs, off_B, off_y, off_p, off_yr, off_t, off_g, off_h;
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
  int t0, T;                  // first 8-row tile, tile count
  int c0, nc;                 // first chunk, chunk count
  int nrg;                    // row groups
};

__device__ __forceinline__ Geo geometry(const TmParams& p) {
  Geo q;
  q.j = (int)cluster_ctarank();
  q.g = (int)blockIdx.x / p.C;
  q.t0 = q.g * p.tiles / p.G;                   // (products stay far below 2^31: tiles <= 2^24, G <= 2^7)
  q.T = (q.g + 1) * p.tiles / p.G - q.t0;
  q.c0 = q.j * p.nch / p.C;
  q.nc = (q.j + 1) * p.nch / p.C - q.c0;
  q.nrg = max(1, (q.T + p.rg_max - 1) / p.rg_max);
  return q;
}

// 8-row tiles [s, s + n) of row group i (an even split).
__device__ __forceinline__ void rg_range(const Geo& q, int i, int& s, int& n) {
  s = i * q.T / q.nrg;
  n = (i + 1) * q.T / q.nrg - s;
}

__device__ __forceinline__ void give_up(int* abort_flag) {
  record_status(&g_dtm_status, DEV_ERR_TIMEOUT);
  atomicExch(abort_flag, 1);
}

// 8 bf16 values (k 0..7 of a group) -> the four (k, k + 4) pairs in MMA order
__device__ __forceinline__ uint4 bf16x8_to_pairs(uint4 v) {
  return make_uint4(__byte_perm(v.x, v.z, 0x5410), __byte_perm(v.x, v.z, 0x7632), __byte_perm(v.y, v.w, 0x5410),
                    __byte_perm(v.y, v.w, 0x7632));
}

// A counter in shared memory published with release and read with acquire
// (CTA scope): the token-sum warp counts the chunks whose sums are written.
__device__ __forceinline__ int ld_acquire_cta(const int* p) {
  int v;
  asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_cta(int* p, int v) {
  asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}

template <int HN>
__device__ __forceinline__ void tmem_ld_n(uint32_t taddr, uint32_t (&r)[HN]) {
  if constexpr (HN == 8) tmem_ld_8cols(taddr, r);
  else if constexpr (HN == 16) tmem_ld_16cols(taddr, r);
  else tmem_ld_32cols(taddr, r);
}

template <int NT, bool PERCH, bool COMP>
__global__ void __launch_bounds__(kThreads, 1)
decode_tm_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                 const __grid_constant__ CUtensorMap tm_a, const TmParams p) {
  // tensor memory columns: A buffers [ABUF][64] at 0, P [NT] after them, then
  // per-group layers: the accumulator ring [DB][NT]; per-channel layers: the
  // slices' sums [SL][NT]
  constexpr int SL = tm_slices(NT, PERCH);
  constexpr int DB = tm_dbufs(NT);
  constexpr int kABufs = tm_abufs(NT);
  constexpr uint32_t kP0 = 64 * kABufs;
  constexpr uint32_t kD0 = kP0 + NT;
  constexpr int HN = NT / 2;                          // token columns of a reduction thread
  static_assert(kD0 + (PERCH ? SL : DB) * NT <= kTmemCols, "tensor memory layout");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_align_up(smem_raw, 1024);
  __shared__ __align__(8) uint64_t full[kMaxStages], empty[kMaxStages], xready[kMaxStages];
  __shared__ __align__(8) uint64_t a_full[kABufs], a_empty[kABufs], d_full[DB], d_empty[DB];
  __shared__ __align__(8) uint64_t acc_full, acc_empty, p_full, ready_bar, done_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort, s_xs_done;

  pdl_launch_dependents();                             // let the next kernel on the stream start queueing
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Geo q = geometry(p);
  const int nst = q.nrg * q.nc;                        // stages of this CTA
  const int n0 = 8 * q.t0;                             // first weight row of the CTA
  float* const xsa = reinterpret_cast<float*>(smem + p.off_xs);   // [chunk][NT] token sums of each chunk
  const bool wg_row = COMP && p.gh == 0;               // the gate row joins the down-projection

  if (threadIdx.x == 0) {
    for (int i = 0; i < p.S; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), kCvt + 1);        // the conversion warps and the MMA commit
      mbar_init(smem_u32(&xready[i]), 1);
    }
    for (int b = 0; b < kABufs; ++b) {
      mbar_init(smem_u32(&a_full[b]), 4);              // the four lane quarters
      mbar_init(smem_u32(&a_empty[b]), 1);
    }
    for (int b = 0; b < DB; ++b) {
      mbar_init(smem_u32(&d_full[b]), 1);
      mbar_init(smem_u32(&d_empty[b]), kRed);
    }
    mbar_init(smem_u32(&acc_full), 1);
    mbar_init(smem_u32(&acc_empty), kRed);
    mbar_init(smem_u32(&p_full), 1);
    mbar_init(smem_u32(&ready_bar), p.C);
    mbar_init(smem_u32(&done_bar), p.C);
    s_abort = 0;
    s_xs_done = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&s_tmem), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  // Cluster barrier, split: every thread arrives now and waits before its
  // first access to another CTA (the row-group epilogue) or before it exits.
  cluster_arrive_relaxed();

  auto slot_base = [&](int s) { return smem + (s % p.S) * p.stage_bytes; };
  auto nbox = [&](int n) { return (8 * n + p.box_rows - 1) / p.box_rows; };
  auto stage_tx = [&](int rg, int n) -> uint32_t {
    uint32_t b = (uint32_t)nbox(n) * p.box_rows * (kChunkK / 2) + NT * kChunkK * 2;
    if (COMP && rg == 0) b += 2 * p.r * 128 + (wg_row ? kChunkK * 2 : 0);
    return b;
  };
  auto slices_of = [&](int rn) { return (8 * rn + 127) / 128; };   // 128-row slices of a row group

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
        rg_range(q, rg, rs, rn);
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
          tma_load_2d(smem_u32(base + p.off_a + p.r * 128), &tm_a, (q.c0 + ch) * kChunkK + 64, 0, bar);
          if (wg_row)
            bulk_load_1d(smem_u32(base + p.off_wg), p.w_g + (size_t)(q.c0 + ch) * kChunkK, kChunkK * 2, bar);
        }
      };
      const int pre = min(p.S, nst);
      // the first stages' codes read only the layer's weights: issued before
      // waiting for the kernel ahead (overlapped launches)
      for (int s = 0; s < pre; ++s) {
        int rs, rn;
        rg_range(q, s / q.nc, rs, rn);
        mbar_arrive_expect_tx(smem_u32(&full[s]), stage_tx(s / q.nc, rn));
        issue_w(s);
      }
      pdl_wait();                                      // tokens may come from the kernel ahead
      for (int s = 0; s < pre; ++s) issue_rest(s);
      issued = pre;
      for (int s = pre; s < nst; ++s) {
        ok = mbar_wait(smem_u32(&empty[s % p.S]), ((s / p.S) & 1) ^ 1, p.wait_ns) && !s_abort;
        if (!ok) break;
        int rs, rn;
        rg_range(q, s / q.nc, rs, rn);
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
    // ------------- token chunk -> the MMA's B layout (+ the chunk's token sums)
    bool ok = true;
    for (int s = 0; s < nst && ok; ++s) {
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&full[s % p.S]), (s / p.S) & 1, p.wait_ns) && !s_abort);
      if (!ok) break;
      const uint8_t* xs = slot_base(s) + p.off_x;
      uint8_t* xb = slot_base(s) + p.off_xb;
      // unit e = e0 + lane: token n = e / 16, 8-k group u16 = e % 16 (panel
      // u16 / 8); a lane keeps its u16 and takes every other token
      if (s < q.nc) {                                  // the first row group covers every chunk once: sums too
#pragma unroll
        for (int i0 = 0; i0 < NT / 2; i0 += 8) {
          float part[8];
#pragma unroll
          for (int ii = 0; ii < 8; ++ii) {
            const int e = 32 * (i0 + ii) + lane, n = e >> 4, u16 = e & 15, pn = u16 >> 3, u = u16 & 7;
            const uint4 v = *reinterpret_cast<const uint4*>(xs + n * (kChunkK * 2) + u16 * 16);
            *reinterpret_cast<uint4*>(xb + pn * NT * 128 + n * 128 + ((u ^ (n & 7)) << 4)) = bf16x8_to_pairs(v);
            part[ii] = ((bf16x2_lo(v.x) + bf16x2_hi(v.x)) + (bf16x2_lo(v.y) + bf16x2_hi(v.y))) +
                       ((bf16x2_lo(v.z) + bf16x2_hi(v.z)) + (bf16x2_lo(v.w) + bf16x2_hi(v.w)));
          }
          // sum over the 16 lanes of a token: independent chains, one per token pair
#pragma unroll
          for (int o = 1; o < 16; o <<= 1)
#pragma unroll
            for (int ii = 0; ii < 8; ++ii) part[ii] += __shfl_xor_sync(0xffffffffu, part[ii], o);
          if ((lane & 15) == 0) {
#pragma unroll
            for (int ii = 0; ii < 8; ++ii) xsa[s * NT + 2 * (i0 + ii) + (lane >> 4)] = part[ii];
          }
        }
      } else {
#pragma unroll 8
        for (int it = 0; it < NT / 2; ++it) {
          const int e = 32 * it + lane, n = e >> 4, u16 = e & 15, pn = u16 >> 3, u = u16 & 7;
          const uint4 v = *reinterpret_cast<const uint4*>(xs + n * (kChunkK * 2) + u16 * 16);
          *reinterpret_cast<uint4*>(xb + pn * NT * 128 + n * 128 + ((u ^ (n & 7)) << 4)) = bf16x8_to_pairs(v);
        }
      }
      fence_proxy_async_smem();                        // the tensor core reads the B layout
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&xready[s % p.S]));
        if (s < q.nc) st_release_cta(&s_xs_done, s + 1);
      }
    }
    if (!ok) give_up(&s_abort);
    cluster_wait();
    return;
  }

  if (warp == kMmaWarp) {
    // ------------------------------------------------------------- MMA
    // (the whole warp runs the loop; one elected lane issues)
    const uint32_t idesc = idesc_bf16_f32(128, NT);
    bool ok = true;
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      ok = __all_sync(0xffffffffu, ok && !s_abort && mbar_wait(smem_u32(bar), parity, p.wait_ns));
    };
    int pc = 0, mc = 0;                                // pairs, per-chunk accumulators issued
    int stage = 0;
    for (int rg = 0; rg < q.nrg && ok; ++rg) {
      int rs, rn;
      rg_range(q, rg, rs, rn);
      const int nsl = slices_of(rn);
      const int npair = nsl + ((COMP && rg == 0) ? 1 : 0);
      // per-channel layers: the sums of the previous row group have been read
      if (PERCH && rg > 0) wait(&acc_empty, (rg - 1) & 1);
      for (int ch = 0; ch < q.nc && ok; ++ch, ++stage) {
        const int slot = stage % p.S;
        wait(&xready[slot], (stage / p.S) & 1);
        const uint32_t xb = smem_u32(slot_base(stage) + p.off_xb);
        for (int i = 0; i < npair && ok; ++i) {
          const bool comp_pair = i == nsl;
          const int ab = pc % kABufs, db = mc % DB;
          wait(&a_full[ab], (pc / kABufs) & 1);
          if (!PERCH && !comp_pair && mc >= DB) wait(&d_empty[db], ((mc / DB) & 1) ^ 1);
          if (!ok) break;
          tc_fence_after();
          const uint32_t d = comp_pair ? tmem + kP0 : PERCH ? tmem + kD0 + NT * i : tmem + kD0 + NT * db;
          const bool over_chunks = comp_pair || PERCH;   // accumulates over the K slice
#pragma unroll
          for (int kk = 0; kk < kChunkK / 16; ++kk) {
            const uint64_t bd = smem_desc(xb + (kk >> 2) * NT * 128 + (kk & 3) * 32, 1024, LAYOUT_SW128);
            const uint32_t acc = (kk > 0 || (over_chunks && ch > 0)) ? 1u : 0u;
            mma_bf16_ts_warp(d, tmem + 64 * ab + 8 * kk, bd, idesc, acc);
          }
          mma_commit_warp(smem_u32(&a_empty[ab]));
          if (!PERCH && !comp_pair) {
            mma_commit_warp(smem_u32(&d_full[db]));
            ++mc;
          }
          ++pc;
        }
        if (ok) mma_commit_warp(smem_u32(&empty[slot]));   // this stage's token layout is no longer read
      }
      if (ok && PERCH) mma_commit_warp(smem_u32(&acc_full));
      if (ok && COMP && rg == 0) mma_commit_warp(smem_u32(&p_full));
    }
    if (!ok && lane == 0) give_up(&s_abort);
    __syncwarp();
    // tensor memory is freed after the conversion and reduction warps' last accesses
    named_sync(2, (kCvt + kRed + 1) * 32);
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
    cluster_wait();
    return;
  }

  if (warp < kCvt) {
    // ------------------------------------------------------ conversion
    const int qd = warp & 3, set = warp >> 2;          // TMEM lane quarter; pairs i with i % kSets == set
    const int lr = 32 * qd + lane;                     // row of a 128-row slice (TMEM lane)
    const uint32_t tl = tmem + ((uint32_t)(32 * qd) << 16);
    bool ok = true;
    auto wait_local = [&](uint64_t* bar, uint32_t parity) {
      ok = __all_sync(0xffffffffu, ok && !s_abort && mbar_wait(smem_u32(bar), parity, p.wait_ns));
    };
    int stage = 0, pc = 0;
    for (int rg = 0; rg < q.nrg; ++rg) {
      int rs, rn;
      rg_range(q, rg, rs, rn);
      const int rows = 8 * rn;
      const int nsl = slices_of(rn);
      const int npair = nsl + ((COMP && rg == 0) ? 1 : 0);
      for (int ch = 0; ch < q.nc; ++ch, ++stage) {
        const int slot = stage % p.S;
        wait_local(&full[slot], (stage / p.S) & 1);
        const uint8_t* base = slot_base(stage);
        for (int i = 0; i < npair; ++i, ++pc) {
          if (pc % kSets != set) continue;
          const int ab = pc % kABufs;
          if (pc >= kABufs) wait_local(&a_empty[ab], ((pc / kABufs) & 1) ^ 1);
          // a lane quarter past the group's rows (or past row r of [A; w_g])
          // is left as it is: those accumulator rows are never read
          const bool idle = i < nsl ? 128 * i + 32 * qd >= rows : 32 * qd > p.r;
          if (ok && !idle) {
            const uint32_t ta = tl + 64 * ab;
            if (i < nsl) {
              // row 128 i + lr of the group (rows past the group repeat its
              // last one; their sums are never stored): its 64-byte chunk
              // row, 16-byte unit u at u ^ ((w >> 1) & 3) (64-byte swizzle:
              // the 8 lanes of a phase hit 8 bank groups)
              const int w = min(128 * i + lr, rows - 1);
              const uint8_t* wrow = base + w * 64;
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                uint32_t v[32];
#pragma unroll
                for (int uu = 0; uu < 2; ++uu) {
                  const int u = 2 * hh + uu;
                  const uint4 wv = *reinterpret_cast<const uint4*>(wrow + ((u ^ ((w >> 1) & 3)) << 4));
                  const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                  for (int k = 0; k < 4; ++k) {
                    uint32_t o[4];
                    nibbles_to_bf16x2_biased(words[k], o);   // 128 + u, pairs (k, k + 4)
#pragma unroll
                    for (int e = 0; e < 4; ++e) v[16 * uu + 4 * k + e] = o[e];
                  }
                }
                tmem_st_32cols(ta + 32 * hh, v);
              }
            } else {
              // row lr of [A; w_g]: 128 bf16 from the stage's two 128-byte
              // swizzled panels of A rows, or the gate row
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                uint32_t v[32];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                  uint4 av = make_uint4(0, 0, 0, 0);
                  if (lr < p.r)
                    av = *reinterpret_cast<const uint4*>(base + p.off_a + hh * p.r * 128 + lr * 128 +
                                                         ((u ^ (lr & 7)) << 4));
                  else if (lr == p.r && wg_row)
                    av = *reinterpret_cast<const uint4*>(base + p.off_wg + hh * 128 + u * 16);
                  const uint4 pr = bf16x8_to_pairs(av);
                  v[4 * u + 0] = pr.x;
                  v[4 * u + 1] = pr.y;
                  v[4 * u + 2] = pr.z;
                  v[4 * u + 3] = pr.w;
                }
                tmem_st_32cols(ta + 32 * hh, v);
              }
            }
            tmem_st_wait();
            tc_fence_before();
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&a_full[ab]));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[slot]));
      }
    }
    if (!ok) give_up(&s_abort);
    tc_fence_before();
    named_sync(2, (kCvt + kRed + 1) * 32);
    cluster_wait();
    return;
  }

  // ------------------------------------------- reduction + epilogue warps
  const int rw = warp - kCvt;                          // 0 .. kRed - 1
  const int tid = threadIdx.x - kCvt * 32;             // 0 .. kRedThreads - 1
  const int qd = rw & 3, hf = rw >> 2;                 // TMEM lane quarter, half of the tokens
  const int lr = 32 * qd + lane;                       // row of a 128-row slice (TMEM lane)
  const uint32_t tl = tmem + ((uint32_t)(32 * qd) << 16);
  __half* const sc_s = reinterpret_cast<__half*>(smem + p.off_sc);   // [8 T][sc_cols] the CTA's scales
  uint8_t* const z_s = smem + p.off_z;                                // [8 T][z_cols] its zero-point bytes
  const int sc0 = q.c0 & ~1;                           // first staged scale column
  const int zb0 = PERCH ? 0 : (q.c0 / 2) & ~3;         // first staged zero-point byte
  const int zrow = (p.ng + 1) / 2;
  __nv_bfloat16* B_s = reinterpret_cast<__nv_bfloat16*>(smem + p.off_B);
  float* ybuf = reinterpret_cast<float*>(smem + p.off_y);     // [rg rows][NT] own partial
  float* pbuf = reinterpret_cast<float*>(smem + p.off_p);     // [r + 1][NT] own partial of P
  float* yred = reinterpret_cast<float*>(smem + p.off_yr);    // [owned rows][NT] cluster sums
  float* tfull = reinterpret_cast<float*>(smem + p.off_t);    // [r + 1][NT] P
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
        for (int e = tid; e < nrow / 2; e += kRedThreads) cp_async4(sc_s + 2 * e, p.scales + (size_t)n0 + 2 * e);
      } else {
        const int pairs = p.sc_cols / 2;
        for (int e = tid; e < nrow * pairs; e += kRedThreads) {
          const int row = e / pairs, col = sc0 + 2 * (e % pairs);
          if (col < p.ng) cp_async4(sc_s + row * p.sc_cols + (col - sc0), p.scales + (size_t)(n0 + row) * p.ng + col);
        }
      }
      if (!p.sym) {
        const int quads = p.z_cols / 4;
        for (int e = tid; e < nrow * quads; e += kRedThreads) {
          const int row = e / quads, col = zb0 + 4 * (e % quads);
          if (col < zrow) cp_async4(z_s + row * p.z_cols + (col - zb0), p.zeros + (size_t)(n0 + row) * zrow + col);
        }
      }
    } else {
      const int cols = p.sc_cols;
      for (int e0 = tid; e0 < nrow * cols; e0 += 8 * kRedThreads) {
        __half v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int e = e0 + u * kRedThreads;
          const int row = e / cols, col = PERCH ? e % cols : sc0 + e % cols;
          v[u] = (e < nrow * cols && col < p.ng) ? p.scales[(size_t)(n0 + row) * p.ng + col] : __half();
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (e0 + u * kRedThreads < nrow * cols) sc_s[e0 + u * kRedThreads] = v[u];
      }
      if (!p.sym) {
        const int zc = p.z_cols;
        for (int e0 = tid; e0 < nrow * zc; e0 += 8 * kRedThreads) {
          uint8_t v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int e = e0 + u * kRedThreads;
            const int row = e / zc, col = zb0 + e % zc;
            v[u] = (e < nrow * zc && col < zrow) ? p.zeros[(size_t)(n0 + row) * zrow + col] : 0;
          }
#pragma unroll
          for (int u = 0; u < 8; ++u)
            if (e0 + u * kRedThreads < nrow * zc) z_s[e0 + u * kRedThreads] = v[u];
        }
      }
    }
    cp_async_commit();                                 // group: scales and zero points
  }
  if (COMP && p.gh > 0) stage_gate_weights_async(p.gw1, p.gw2, p.gc1, p.gc2, p.r, p.gh, gate_s, tid, kRedThreads);
  else cp_async_commit();                              // (an empty group keeps the count)
  pdl_wait();                                          // y follows the kernel ahead

  bool ok = true;
  auto wait_local = [&](uint64_t* bar, uint32_t parity) {
    ok = __all_sync(0xffffffffu, ok && !s_abort && mbar_wait(smem_u32(bar), parity, p.wait_ns));
  };
  auto wait_cluster = [&](uint64_t* bar, uint32_t parity) {
    ok = __all_sync(0xffffffffu, ok && !s_abort && mbar_wait_cluster(smem_u32(bar), parity, p.wait_ns));
  };
  // the token sums of chunks [0, n) are written (bounded wait)
  auto wait_sums = [&](int n) {
    bool done = ld_acquire_cta(&s_xs_done) >= n;
    if (!done && ok) {
      const uint64_t t0 = globaltimer_ns();
      while (!(done = ld_acquire_cta(&s_xs_done) >= n) && !s_abort && globaltimer_ns() - t0 <= p.wait_ns)
        __nanosleep(32);
    }
    ok = __all_sync(0xffffffffu, ok && done);
  };

  int red_mc = 0;                                      // per-chunk accumulators reduced
  bool cluster_ready = false;
  for (int rg = 0; rg < q.nrg; ++rg) {
    int rs, rn;
    rg_range(q, rg, rs, rn);
    const int rows = 8 * rn;                           // rows of the row group
    const int nsl = slices_of(rn);
    const int o0 = 8 * (q.j * rn / p.C), o1 = 8 * ((q.j + 1) * rn / p.C);   // rows finished here
    // peers have finished reading this CTA's partial of the previous row group
    if (rg > 0) wait_cluster(&done_bar, (rg - 1) & 1);
    // the factor-B rows of the rows finished here (contiguous in B)
    if (COMP) {
      const int per = p.r / 8;                         // 16-byte pieces per row
      const int nb = (o1 - o0) * per;
      for (int e = tid; e < nb; e += kRedThreads)
        cp_async16(B_s + (size_t)e * 8, p.B + (size_t)(n0 + 8 * rs + o0) * p.r + (size_t)e * 8);
    }
    cp_async_commit();                                 // group: this row group's B rows
    if (rg == 0) {
      cp_async_wait<2>();                              // the scales and zero points
      named_sync(1, kRedThreads);
    }

    // ------------------------------- this CTA's partial -> shared memory [row][NT]
    if constexpr (!PERCH) {
      float acc[SL][HN];
#pragma unroll
      for (int sl = 0; sl < SL; ++sl)
#pragma unroll
        for (int j = 0; j < HN; ++j) acc[sl][j] = 0.0f;
      for (int ch = 0; ch < q.nc; ++ch) {
        if (rg == 0) wait_sums(ch + 1);
        const float4* xs4 = reinterpret_cast<const float4*>(xsa + ch * NT + hf * HN);
        const int chg = q.c0 + ch;
#pragma unroll
        for (int sl = 0; sl < SL; ++sl) {
          if (sl < nsl) {
            const int db = red_mc % DB;
            wait_local(&d_full[db], (red_mc / DB) & 1);
            // S += s D - (128 + z) s sum_k x, per row and chunk (D read in
            // pieces of at most 16 columns)
            constexpr int PC = HN < 16 ? HN : 16;
            const int rc = 8 * rs + min(128 * sl + lr, rows - 1);   // row of the CTA
            const float sv = __half2float(sc_s[rc * p.sc_cols + chg - sc0]);
            const int z = p.sym ? 8 : (z_s[rc * p.z_cols + chg / 2 - zb0] >> (4 * (chg & 1))) & 15;
            const float zs = -(float)(128 + z) * sv;
            if (ok) tc_fence_after();
#pragma unroll
            for (int c0 = 0; c0 < HN; c0 += PC) {
              uint32_t dv[PC];
              if (ok) {
                tmem_ld_n<PC>(tl + kD0 + NT * db + hf * HN + c0, dv);
                tmem_ld_wait();
#pragma unroll
                for (int j4 = 0; j4 < PC / 4; ++j4) {
                  const float4 xv = xs4[c0 / 4 + j4];
                  const int j = c0 + 4 * j4;
                  acc[sl][j + 0] = fmaf(sv, __uint_as_float(dv[4 * j4 + 0]), fmaf(zs, xv.x, acc[sl][j + 0]));
                  acc[sl][j + 1] = fmaf(sv, __uint_as_float(dv[4 * j4 + 1]), fmaf(zs, xv.y, acc[sl][j + 1]));
                  acc[sl][j + 2] = fmaf(sv, __uint_as_float(dv[4 * j4 + 2]), fmaf(zs, xv.z, acc[sl][j + 2]));
                  acc[sl][j + 3] = fmaf(sv, __uint_as_float(dv[4 * j4 + 3]), fmaf(zs, xv.w, acc[sl][j + 3]));
                }
              }
            }
            if (ok) tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&d_empty[db]));
            ++red_mc;
          }
        }
      }
#pragma unroll
      for (int sl = 0; sl < SL; ++sl) {
        const int row = 128 * sl + lr;
        if (sl < nsl && row < rows) {
#pragma unroll
          for (int j = 0; j < HN; j += 4)
            *reinterpret_cast<float4*>(ybuf + (size_t)row * NT + hf * HN + j) =
                make_float4(acc[sl][j], acc[sl][j + 1], acc[sl][j + 2], acc[sl][j + 3]);
        }
      }
    } else {
      // per-channel layers: S - (128 + z) (sum of x over the K slice), in
      // pieces of 8 token columns
      wait_local(&acc_full, rg & 1);
      if (rg == 0) wait_sums(q.nc);
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < HN; c0 += 8) {
          float xt[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) xt[j] = 0.0f;
          for (int ch = 0; ch < q.nc; ++ch) {
            const float4* xs4 = reinterpret_cast<const float4*>(xsa + ch * NT + hf * HN + c0);
            const float4 a = xs4[0], b = xs4[1];
            xt[0] += a.x; xt[1] += a.y; xt[2] += a.z; xt[3] += a.w;
            xt[4] += b.x; xt[5] += b.y; xt[6] += b.z; xt[7] += b.w;
          }
#pragma unroll
          for (int sl = 0; sl < SL; ++sl) {
            if (sl < nsl) {
              uint32_t av[8];
              tmem_ld_8cols(tl + kD0 + NT * sl + hf * HN + c0, av);
              tmem_ld_wait();
              const int row = 128 * sl + lr;
              if (row < rows) {
                const float zt = -(float)(128 + (p.sym ? 8 : (z_s[(8 * rs + row) * p.z_cols] & 15)));
                float* yo = ybuf + (size_t)row * NT + hf * HN + c0;
                *reinterpret_cast<float4*>(yo) =
                    make_float4(fmaf(zt, xt[0], __uint_as_float(av[0])), fmaf(zt, xt[1], __uint_as_float(av[1])),
                                fmaf(zt, xt[2], __uint_as_float(av[2])), fmaf(zt, xt[3], __uint_as_float(av[3])));
                *reinterpret_cast<float4*>(yo + 4) =
                    make_float4(fmaf(zt, xt[4], __uint_as_float(av[4])), fmaf(zt, xt[5], __uint_as_float(av[5])),
                                fmaf(zt, xt[6], __uint_as_float(av[6])), fmaf(zt, xt[7], __uint_as_float(av[7])));
              }
            }
          }
        }
        tc_fence_before();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&acc_empty));   // the next row group's MMAs may overwrite the sums
    }
    if (COMP && rg == 0) {
      // this CTA's partial of P = [A; w_g] x over its K slice (tcgen05.ld is
      // warp-collective: lanes past row r join a load they discard)
      wait_local(&p_full, 0);
      if (ok) {
        tc_fence_after();
        uint32_t av[HN];
        tmem_ld_n<HN>(tl + kP0 + hf * HN, av);
        tmem_ld_wait();
        if (lr <= p.r) {
#pragma unroll
          for (int j = 0; j < HN; j += 4)
            *reinterpret_cast<float4*>(pbuf + (size_t)lr * NT + hf * HN + j) =
                make_float4(__uint_as_float(av[j]), __uint_as_float(av[j + 1]), __uint_as_float(av[j + 2]),
                            __uint_as_float(av[j + 3]));
        }
        tc_fence_before();
      }
    }

    // ------------------------------------------ row-group epilogue (cluster)
    named_sync(1, kRedThreads);
    if (!cluster_ready) {                              // every peer's barriers are initialised
      cluster_wait();
      cluster_ready = true;
    }
    // one lane per peer: the arrives (release, cluster scope) go out together
    if (rw == 0 && lane < p.C && ok && !s_abort) mbar_arrive_remote(dsmem_addr(smem_u32(&ready_bar), (uint32_t)lane));
    wait_cluster(&ready_bar, rg & 1);

    // every CTA's partials are in place: sum P (first row group) and this
    // CTA's rows over the cluster, in rank order, four loads in flight
    const int nown = o1 - o0;
    if (ok) {
      const int pu = (COMP && rg == 0) ? (p.r + 1) * NT / 4 : 0;       // float4 units of P
      const int yu = nown * NT / 4;                                     // float4 units of owned rows
      const uint32_t pb = smem_u32(pbuf), yb = smem_u32(ybuf) + (uint32_t)o0 * NT * 4;
      for (int e = tid; e < pu + yu; e += kRedThreads) {
        const uint32_t la = e < pu ? pb + (uint32_t)e * 16 : yb + (uint32_t)(e - pu) * 16;
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
        if (e < pu) reinterpret_cast<float4*>(tfull)[e] = sum;           // P [r + 1][NT]
        else reinterpret_cast<float4*>(yred)[e - pu] = sum;              // [owned rows][NT]
      }
    }
    named_sync(1, kRedThreads);
    // this CTA's reads of the peers' partials are done
    if (rw == 0 && lane < p.C && ok && !s_abort) mbar_arrive_remote(dsmem_addr(smem_u32(&done_bar), (uint32_t)lane));

    float* Tm = hid_s + (p.gh > 0 ? NT * gate_hid_stride(p.gh) : 0);   // T [NT][r] (after the hidden units)
    if (COMP && rg == 0 && ok) {
      const int rk = p.r;
      if (p.gh > 0) {
        cp_async_wait<1>();                            // the staged gate weights (the B rows may still land)
        named_sync(1, kRedThreads);
        // vector gate over all tokens: t [NT][r] = P[0..r)^T
        for (int e = tid; e < NT * rk; e += kRedThreads) Tm[e] = tfull[(e % rk) * NT + e / rk];
        named_sync(1, kRedThreads);
        const GateSmem gt(gate_s, rk, p.gh);
        vector_gate_hidden_rows(Tm, NT, gt, hid_s, tid, kRedThreads);
        named_sync(1, kRedThreads);
        vector_gate_apply_rows(Tm, NT, gt, hid_s, tid, kRedThreads);
        named_sync(1, kRedThreads);
        for (int e = tid; e < NT * rk; e += kRedThreads) Tm[e] = (e / rk < p.M) ? p.alpha * Tm[e] : 0.0f;
      } else {
        for (int e = tid; e < NT * rk; e += kRedThreads) {
          const int m = e / rk, i = e % rk;
          const float gm = m < p.M ? p.alpha / (1.0f + expf(-(tfull[rk * NT + m] + p.b_g))) : 0.0f;
          Tm[e] = gm * tfull[i * NT + m];
        }
      }
    }
    cp_async_wait<0>();                                // the factor-B rows
    named_sync(1, kRedThreads);

    // y for the rows finished here: one (row, token) element per thread and
    // step, rows fastest (coalesced stores); the correction sum_j B[n][j] T[m][j]
    if (ok) {
      for (int e = tid; e < nown * p.M; e += kRedThreads) {
        const int rr = e % nown, m = e / nown;
        const int rc = 8 * rs + o0 + rr;               // row of the CTA
        float v = yred[rr * NT + m];
        if (PERCH) v *= __half2float(sc_s[rc * p.sc_cols]);
        if (COMP) {
          const __nv_bfloat162* brow = reinterpret_cast<const __nv_bfloat162*>(B_s + (size_t)rr * p.r);
          const float* tr = Tm + m * p.r;
          float c0 = 0.0f, c1 = 0.0f;
          for (int jj = 0; jj < p.r / 2; ++jj) {
            const float2 bb = __bfloat1622float2(brow[jj]);
            c0 = fmaf(bb.x, tr[2 * jj], c0);
            c1 = fmaf(bb.y, tr[2 * jj + 1], c1);
          }
          v += c0 + c1;
        }
        const size_t o = (size_t)m * p.N + n0 + rc;
        if (p.out_f32) reinterpret_cast<float*>(p.y)[o] = v;
        else reinterpret_cast<__nv_bfloat16*>(p.y)[o] = __float2bfloat16_rn(v);
      }
    }
    named_sync(1, kRedThreads);                        // B rows / partial buffers are reused by the next row group
  }
  // peers are done reading this CTA's shared memory (and arriving on its
  // barriers) before it exits: waited for even after a failure, bounded
  if (!mbar_wait_cluster(smem_u32(&done_bar), (q.nrg - 1) & 1, p.wait_ns)) ok = false;
  if (!ok) give_up(&s_abort);
  // the MMA warp frees tensor memory once every conversion and reduction
  // warp is past its last access
  tc_fence_before();
  named_sync(2, (kCvt + kRed + 1) * 32);
}

using TmKernel = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, TmParams);

template <int NT>
TmKernel pick_nt(bool perch, bool comp) {
  if (perch) return comp ? decode_tm_kernel<NT, true, true> : decode_tm_kernel<NT, true, false>;
  return comp ? decode_tm_kernel<NT, false, true> : decode_tm_kernel<NT, false, false>;
}

TmKernel pick_tm(int NT, bool perch, bool comp) {
  return NT == 16 ? pick_nt<16>(perch, comp) : NT == 32 ? pick_nt<32>(perch, comp) : pick_nt<64>(perch, comp);
}

// ---------------------------------------------------------------- plan --
struct TmPlan {
  int device, N, K, G, rank, comp, NT, gh, sym;   // key
  int C, Gc, tiles, nch, rg_max, S, box_rows, meta_async;
  size_t smem;
  uint32_t stage_bytes, off_x, off_xb, off_a, off_wg;
  uint32_t off_sc, off_z, off_xs, off_B, off_y, off_p, off_yr, off_t, off_g, off_h;
  int sc_cols, z_cols;
  TmKernel fn;
};

size_t up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Shared-memory layout for `rg_max` tiles per row group, S stages, the
// scales / zero points of `meta_rows` rows and the token sums of `nc_max`
// chunks; (size_t)-1 if an alignment rule would break.
size_t layout(TmPlan* c, int rg_max, int S, int NT, int rank, int ncs_max, int nzs_max, int meta_rows, int nc_max) {
  const int rows = 8 * rg_max;
  const int nb = (rows + kMaxBoxRows - 1) / kMaxBoxRows;
  c->box_rows = 8 * ((rows / 8 + nb - 1) / nb);
  size_t st = (size_t)nb * c->box_rows * (kChunkK / 2);
  st = up(st, 1024);
  c->off_x = (uint32_t)st;                        // raw token chunk (TMA)
  st = up(st + (size_t)NT * kChunkK * 2, 1024);
  c->off_xb = (uint32_t)st;                       // tokens in the MMA's layout (two 1024-aligned panels)
  st += (size_t)2 * NT * 128;
  c->off_a = (uint32_t)st;                        // rows of A: two 128-byte swizzled panels
  st += (size_t)2 * std::max(rank, 8) * 128;
  c->off_wg = (uint32_t)st;                       // w_g
  st += (size_t)kChunkK * 2;
  c->stage_bytes = (uint32_t)up(st, 1024);
  // TMA destinations: codes (64-byte swizzle: 512-byte aligned boxes), tokens,
  // A panels (128-byte swizzle: 1024-byte aligned), w_g (16 bytes)
  if ((c->box_rows * (kChunkK / 2)) % 512 != 0 || c->off_x % 128 || c->off_xb % 1024 || (NT * 128) % 1024 ||
      c->off_a % 1024 || (rank * 128) % 1024 || c->off_wg % 16)
    return (size_t)-1;
  size_t off = (size_t)S * c->stage_bytes;
  c->off_sc = (uint32_t)off;                     // the CTA's scales and zero points
  off = up(off + (size_t)meta_rows * ncs_max * 2, 16);
  c->off_z = (uint32_t)off;
  off = up(off + (size_t)meta_rows * nzs_max, 16);
  c->off_xs = (uint32_t)off;                     // token sums [chunk][NT]
  off = up(off + (size_t)nc_max * NT * 4, 16);
  const int own_rows = 8 * ((rg_max + c->C - 1) / c->C + 1);
  c->off_B = (uint32_t)off;
  off = up(off + (size_t)own_rows * std::max(rank, 8) * 2, 16);
  c->off_y = (uint32_t)off;
  off = up(off + (size_t)rows * NT * 4, 16);
  c->off_p = (uint32_t)off;
  off = up(off + (size_t)(rank + 1) * NT * 4, 16);
  c->off_yr = (uint32_t)off;
  off = up(off + (size_t)own_rows * NT * 4, 16);
  c->off_t = (uint32_t)off;
  off = up(off + (size_t)(rank + 1) * NT * 4, 16);
  c->off_g = (uint32_t)off;
  off = up(off + (c->gh > 0 ? (size_t)gate_smem_floats(rank, c->gh) * 4 : 0), 16);
  c->off_h = (uint32_t)off;                       // hidden units (vector gate), then T [NT][r]
  off = up(off + (c->gh > 0 ? (size_t)NT * gate_hid_stride(c->gh) * 4 : 0) + (size_t)NT * std::max(rank, 1) * 4, 16);
  return off + 1024;                             // alignment slack of the dynamic base
}

int env_int(const char* name, int dflt) {
  const char* v = std::getenv(name);
  return (v && v[0]) ? std::atoi(v) : dflt;
}

int build_tm_plan(const spear_w4_layer& L, int NT, bool comp, const DeviceInfo& di, TmPlan* pl) {
  const bool perch = L.group_size == L.K;
  pl->NT = NT;
  pl->fn = pick_tm(NT, perch, comp);
  pl->tiles = L.N / 8;
  pl->nch = L.K / kChunkK;
  int C = env_int("SPEAR_DECODE_CLUSTER", 8);
  C = std::max(1, std::min(C, kMaxC));
  while (C > 1 && pl->nch < C) C /= 2;
  pl->C = C;

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
  // clusters: as many as fit at one CTA per SM (all tensor memory is taken)
  cfg.gridDim = dim3(C);
  cfg.dynamicSmemBytes = optin;
  int max_clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&max_clusters, pl->fn, &cfg) != cudaSuccess || max_clusters < 1) {
    cudaGetLastError();
    return fail(SPEAR_ERR_UNSUPPORTED, "decode: no cluster of %d CTAs fits", C);
  }
  int Gc = env_int("SPEAR_DECODE_CLUSTERS", max_clusters);
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

  // row groups: the fewest that fit (at most tm_slices slices of 128 rows each)
  const int rg_top = std::min(tm_slices(NT, perch) * 16, T_max);
  bool found = false;
  for (int nrg = 1; nrg <= 1024 && !found; ++nrg) {
    const int rg = (T_max + nrg - 1) / nrg;
    if (rg > rg_top) continue;
    for (int S = kMaxStages; S >= 2 && !found; --S) {
      TmPlan c = *pl;
      const size_t sm = layout(&c, rg, S, NT, L.rank, ncs_max, nzs_max, 8 * T_max, c_per);
      if (sm <= optin) {
        c.rg_max = rg;
        c.S = S;
        c.smem = sm;
        c.sc_cols = ncs_max;
        c.z_cols = nzs_max;
        *pl = c;
        found = true;
      }
    }
    if (rg == 1) break;
  }
  if (!found) return fail(SPEAR_ERR_UNSUPPORTED, "decode: no shared-memory layout for N=%d K=%d", L.N, L.K);
  return SPEAR_OK;
}

int get_tm_plan(const spear_w4_layer& L, int M, TmPlan* out) {
  DeviceInfo di;
  if (int rc = device_info(&di)) return rc;
  const int NT = M <= 16 ? 16 : M <= 32 ? 32 : 64;
  const int comp = (L.comp_enabled && L.rank > 0) ? 1 : 0;
  const int gh = comp ? L.gate_hidden : 0;
  static std::mutex mu;
  static std::vector<TmPlan> cache;
  std::lock_guard<std::mutex> lk(mu);
  for (const TmPlan& p : cache)
    if (p.device == di.device && p.N == L.N && p.K == L.K && p.G == L.group_size && p.rank == L.rank &&
        p.comp == comp && p.NT == NT && p.gh == gh && p.sym == L.symmetric) {
      *out = p;
      return SPEAR_OK;
    }
  TmPlan p{};
  p.gh = gh;
  if (int rc = build_tm_plan(L, NT, comp != 0, di, &p)) return rc;
  p.device = di.device; p.N = L.N; p.K = L.K; p.G = L.group_size; p.rank = L.rank; p.comp = comp; p.sym = L.symmetric;
  if (log_plans())
    fprintf(stderr, "[spear] decode tm plan N=%d K=%d G=%d rank=%d comp=%d NT=%d: C=%d clusters=%d rg_max=%d S=%d "
            "box_rows=%d stage=%u smem=%zu\n", L.N, L.K, L.group_size, L.rank, comp, NT, p.C, p.Gc, p.rg_max,
            p.S, p.box_rows, p.stage_bytes, p.smem);
  if (cache.size() > 4096) cache.clear();
  cache.push_back(p);
  *out = p;
  return SPEAR_OK;
}


}  // namespace

bool decode_tm_supports(const spear_w4_layer& L, int M) {
  if (M < 1 || M > 64) return false;
  if (!env_int("SPEAR_DECODE_TM", 0)) return false;     // opt-in while it is measured
  TmPlan pl;
  char saved[512];
  snprintf(saved, sizeof(saved), "%s", spear_last_error());
  const int rc = get_tm_plan(L, M, &pl);
  if (rc != SPEAR_OK) set_last_error(saved);
  return rc == SPEAR_OK;
}


int launch_decode_tm(const spear_w4_layer& L, const uint16_t* x, int M, void* y, int out_f32, cudaStream_t st,
                     bool overlap) {
  TmPlan pl;
  if (int rc = get_tm_plan(L, M, &pl)) return rc;
  const int NT = pl.NT;
  const bool comp = pl.comp != 0;
  CUtensorMap tm_w, tm_x, tm_a;
  if (int rc = make_tmap(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, L.qweight, L.K / 2, L.N, kChunkK / 2, pl.box_rows,
                         CU_TENSOR_MAP_SWIZZLE_64B)) return rc;
  if (int rc = make_tmap(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, L.K, M, kChunkK, NT,
                         CU_TENSOR_MAP_SWIZZLE_NONE)) return rc;
  if (comp) {
    if (int rc = make_tmap(&tm_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, L.A, L.K, L.rank, 64, L.rank,
                           CU_TENSOR_MAP_SWIZZLE_128B)) return rc;
  } else {
    tm_a = tm_x;                                   // never used
  }
  TmParams p{};
  p.N = L.N; p.K = L.K; p.M = M; p.sym = L.symmetric; p.ng = L.K / L.group_size;
  p.C = pl.C; p.G = pl.Gc; p.tiles = pl.tiles; p.nch = pl.nch;
  p.r = comp ? L.rank : 0;
  p.rg_max = pl.rg_max; p.S = pl.S; p.box_rows = pl.box_rows;
  p.stage_bytes = pl.stage_bytes; p.off_x = pl.off_x; p.off_xb = pl.off_xb; p.off_xs = pl.off_xs;
  p.off_a = pl.off_a; p.off_wg = pl.off_wg;
  p.off_sc = pl.off_sc; p.off_z = pl.off_z; p.off_B = pl.off_B; p.off_y = pl.off_y; p.off_p = pl.off_p;
  p.off_yr = pl.off_yr; p.off_t = pl.off_t; p.off_g = pl.off_g; p.off_h = pl.off_h;
  p.sc_cols = pl.sc_cols; p.z_cols = pl.z_cols; p.meta_async = pl.meta_async;
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

int read_and_clear_status_decode_tm(unsigned* out, cudaStream_t st) {
  void* addr = nullptr;
  if (int rc = cuda_check(cudaGetSymbolAddress(&addr, g_dtm_status), "decode status address")) return rc;
  if (int rc = cuda_check(cudaMemcpyAsync(out, addr, sizeof(unsigned), cudaMemcpyDeviceToHost, st),
                          "read decode status")) return rc;
  if (int rc = cuda_check(cudaStreamSynchronize(st), "read decode status")) return rc;
  return cuda_check(cudaMemsetAsync(addr, 0, sizeof(unsigned), st), "clear decode status");
}

}  // namespace spear
