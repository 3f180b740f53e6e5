// prefill.cu -- prefill path of the gated W4 + low-rank compensated linear
// (SPEAR explainer, Technical Summary 2.2 A: prefill is compute-bound; the
// compensator runs as a separate kernel next to the GEMM instead of inside it).
//
// Kernels
//  * w4_gemm_tc: Y[M][N] = X[M][K] * dequant(Wq)^T on the 5th-generation tensor
//    cores, fp16 operands, fp32 accumulation.  One 128- or 256-token x 256
//    (outputs) tile per thread block; K in steps of 64.  A TMA warp loads the
//    fp16 copy of the X tile (128-byte swizzle) and the raw int4 tile; eight
//    converter warps expand the int4 tile to fp16 straight into the tensor
//    core's swizzled K-major layout; one thread issues tcgen05.mma into fp32
//    accumulators in tensor memory; the same eight warps then drain them
//    (tcgen05.ld) and store Y.
//      - per-channel scales: the tile holds the exact integers (u - z) and the
//        fp32 scale of each output column is applied in the epilogue;
//      - group scales: the tile holds (u - z) * s rounded once to fp16
//        (11 significant bits: a bf16 operand's 8 bits are not enough when a
//        few outlier channels dominate an output).
//    The activations are bf16; their fp16 copy is exact for |x| < 65504 and
//    is written by the pass that already reads X (comp_down) or by to_fp16,
//    with each 8-k chunk in the order 0,4,1,5,2,6,3,7 -- the order in which
//    the converters take nibble pairs out of a 32-bit word -- so neither side
//    permutes bytes.  Eight converter warps (one weight row per thread) keep
//    the zero points and scales of the next four groups in flight.
//    Optionally ("fused" mode) the K loop is extended by the compensator's
//    up-projection: extra K steps with A = [T_hi | T_lo] (the gated
//    down-projection split into two bf16 halves) and B = the factor B, into a
//    second accumulator that the epilogue adds unscaled.
//    Grids of a few 128-token tiles (small M) split K over a cluster of 2 or
//    4 CTAs: each dequantises its share of the 256-row slab, drains its
//    partial (scaled, with the correction on rank 0) into its own shared
//    memory, and finishes 256 / KS output columns by summing the partials of
//    the cluster in rank order through distributed shared memory.
//  * comp_down: T[m][j] = alpha * g_m * (A x_m)[j], g_m = sigmoid(w_g . x_m + b_g),
//    written as bf16 hi/lo pairs; mma.sync over token tiles, one pass over X.
//  * comp_up_add: Y[m][n] += sum_j T[m][j] B[n][j] in place ("stream" mode:
//    runs after the plain W4 GEMM, while comp_down ran beside it on a second
//    stream).
#include <cuda.h>

#include <algorithm>
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"
#include "tmap.h"

namespace spear {
namespace {

__device__ unsigned g_prefill_status;

using namespace sm100;

constexpr int kBN = 256;                  // outputs per tile (MMA N)
constexpr int kBK = 64;                   // k per stage (one 128-byte swizzle row of bf16)
constexpr int kWBytes = kBN * kBK * 2;    // 32 KB
constexpr int kRawBytes = kBN * kBK / 2;  // 8 KB
constexpr int kGemmThreads = 320;         // warp 0: TMA, warp 1: MMA, warps 2-9: convert + epilogue
constexpr uint32_t kTmemCols = 512;

// BM tokens per tile: 128 (one M = 128 MMA per 16 k; accumulator in TMEM
// columns [0, 256), the fused correction in [256, 512)) or 256 (two M = 128
// MMAs per 16 k on the same converted weight tile, accumulators in [0, 256)
// and [256, 512), the fused correction added into them), which halves the
// dequantisation work and the int4 traffic per output.
template <int BM>
struct TileCfg {
  static constexpr int kStages = BM == 256 ? 3 : 4;
  static constexpr int kXBytes = BM * kBK * 2;          // 16 or 32 KB
  static constexpr int kStageBytes = kXBytes + kWBytes + kRawBytes;
  static constexpr int kMH = BM / 128;                  // M = 128 MMAs per 16 k
};
constexpr uint64_t kWaitNs = 2000ull * 1000 * 1000;   // 2 s: far beyond any legitimate wait

struct GemmParams {
  int M, N, K, G, ng, sym, perch;
  const __half* scales;
  const uint8_t* zeros;
  void* y;
  int out_f32;
  int comp_stages;      // extra K steps of the fused up-projection (0 = none)
  int r;
  int t_row_bytes;      // bytes per T2 row box (<= 128)
  int b_row_bytes;      // bytes per B row (2r)
  int ks;               // CTAs of a cluster splitting K (1, 2 or 4; 128-token tiles only)
  const float* tscale;  // [M] 2^e_m: the fp16 token copy holds x_m 2^-e_m (power-of-two token scaling)
};

// K split: the partial accumulators of a cluster meet in shared memory,
// [128 tokens][256 + 4] fp32 per CTA (16-byte rows, conflict-free)
constexpr int kRedStride = kBN + 4;

__device__ __forceinline__ uint32_t sw_layout(int row_bytes) {
  return row_bytes >= 128 ? LAYOUT_SW128 : row_bytes == 64 ? LAYOUT_SW64 : LAYOUT_SW32;
}

template <int BM>
__global__ void __launch_bounds__(kGemmThreads, 1)
w4_gemm_tc(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_wq,
           const __grid_constant__ CUtensorMap tm_t, const __grid_constant__ CUtensorMap tm_b,
           const GemmParams p) {
  using C = TileCfg<BM>;
  constexpr int kStages = C::kStages, kXBytes = C::kXBytes, kStageBytes = C::kStageBytes, kMH = C::kMH;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align_up(smem_raw, 1024);
  __shared__ __align__(8) uint64_t bar_full[kStages], bar_cvt[kStages], bar_empty[kStages], bar_acc;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kBN, m0 = blockIdx.y * BM;
  const int k_stages = p.K / kBK;
  // K split over a cluster of KS CTAs: this CTA's main K steps are [kb, ke);
  // the fused correction's steps go to rank 0
  const int KS = p.ks;
  const int krank = KS > 1 ? (int)cluster_ctarank() : 0;
  const int kb = (int)((long long)krank * k_stages / KS), ke = (int)((long long)(krank + 1) * k_stages / KS);
  const int nmain = ke - kb;
  const int ncomp = krank == 0 ? p.comp_stages : 0;
  const int total_stages = nmain + ncomp;
  SPEAR_CHECK(&g_prefill_status, 0 <= kb && kb <= ke && ke <= k_stages && krank < KS && n0 < p.N && m0 < p.M);

  auto x_slot = [&](int s) { return smem + s * kStageBytes; };
  auto w_slot = [&](int s) { return smem + s * kStageBytes + kXBytes; };
  auto raw_slot = [&](int s) { return smem + s * kStageBytes + kXBytes + kWBytes; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bar_full[s]), 1);
      mbar_init(smem_u32(&bar_cvt[s]), 8);
      mbar_init(smem_u32(&bar_empty[s]), 1);
    }
    mbar_init(smem_u32(&bar_acc), 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&s_tmem), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_x);
    prefetch_tmap(&tm_wq);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  auto give_up = [&]() {
    record_status(&g_prefill_status, DEV_ERR_TIMEOUT);
    atomicExch(&s_abort, 1);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // The whole warp runs the loop (every lane waits, lane 0 issues): a loop
    // on one lane while the other 31 wait at a barrier runs at about a third
    // of the rate.  The same holds for the MMA issuer below.
    int issued = 0;
    for (int s = 0; s < total_stages; ++s) {
      const int slot = s % kStages;
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_empty[slot]), ((s / kStages) & 1) ^ 1, kWaitNs) &&
                                       !s_abort)) {
        if (lane == 0) give_up();
        break;
      }
      if (lane == 0) {
        const uint32_t full = smem_u32(&bar_full[slot]);
        if (s < nmain) {
          const int sg = kb + s;        // K step
          mbar_arrive_expect_tx(full, kXBytes + kRawBytes);
          tma_load_2d(smem_u32(x_slot(slot)), &tm_x, sg * kBK, m0, full);
          tma_load_2d(smem_u32(raw_slot(slot)), &tm_wq, sg * (kBK / 2), n0, full);
        } else {
          const int j = s - nmain;      // compensator step: T box j and the factor B
          mbar_arrive_expect_tx(full, BM * p.t_row_bytes + kBN * p.b_row_bytes);
          tma_load_2d(smem_u32(x_slot(slot)), &tm_t, j * 64, m0, full);
          tma_load_2d(smem_u32(w_slot(slot)), &tm_b, 0, n0, full);
        }
      }
      __syncwarp();
      ++issued;
    }
    // never leave with copies in flight: wait (bounded) for every issued stage
    if (s_abort && lane == 0) {
      for (int s = std::max(0, issued - kStages); s < issued; ++s)
        mbar_wait(smem_u32(&bar_full[s % kStages]), (s / kStages) & 1, kWaitNs);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    {
      const uint32_t idesc = idesc_f16_f32(128, kBN);            // fp16 X x fp16 W (M = 128 per MMA)
      const uint32_t idesc_comp = idesc_bf16_f32(128, kBN);      // bf16 T x bf16 B
      bool ok = true;
      for (int s = 0; s < total_stages && ok; ++s) {
        const int slot = s % kStages;
        const uint32_t ph = (s / kStages) & 1;
        ok = mbar_wait(smem_u32(&bar_full[slot]), ph, kWaitNs) && !s_abort;
        if (ok && s < nmain) ok = mbar_wait(smem_u32(&bar_cvt[slot]), ph, kWaitNs) && !s_abort;
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) { if (lane == 0) give_up(); break; }
        tc_fence_after();
        const uint32_t xa = smem_u32(x_slot(slot)), wa = smem_u32(w_slot(slot));
        if (s < nmain) {
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint64_t bd = smem_desc(wa + 32 * k, 1024, LAYOUT_SW128);
#pragma unroll
            for (int mh = 0; mh < kMH; ++mh) {                 // token rows 128 mh .. (16 KB apart)
              const uint64_t ad = smem_desc(xa + mh * 16384 + 32 * k, 1024, LAYOUT_SW128);
              mma_bf16_ss_warp(tmem + mh * kBN, ad, bd, idesc, (s > 0 || k > 0) ? 1u : 0u);
            }
          }
        } else {
          // A = T box j (columns 64j.. of [T_hi | T_lo]); B = the factor B (k = rank).
          // BM = 128: accumulated into the second accumulator (columns 256..511);
          // BM = 256 (group scales only): added into the main accumulators.
          const int j = s - nmain;
          const uint32_t a_layout = sw_layout(p.t_row_bytes), b_layout = sw_layout(p.b_row_bytes);
          for (int i = 0; i < p.t_row_bytes / 32; ++i) {
            const int col = 64 * j + 16 * i;                 // column of [T_hi | T_lo]
            if (col >= 2 * p.r) break;
            const int bstep = (col % p.r) / 16;
            const uint64_t bd = smem_desc(wa + 32 * bstep, 8 * p.b_row_bytes, b_layout);
#pragma unroll
            for (int mh = 0; mh < kMH; ++mh) {
              const uint64_t ad = smem_desc(xa + mh * 128 * p.t_row_bytes + 32 * i, 8 * p.t_row_bytes, a_layout);
              if (kMH == 1) mma_bf16_ss_warp(tmem + kBN, ad, bd, idesc_comp, (j > 0 || i > 0) ? 1u : 0u);
              else mma_bf16_ss_warp(tmem + mh * kBN, ad, bd, idesc_comp, 1u);
            }
          }
        }
        mma_commit_warp(smem_u32(&bar_empty[slot]));        // frees the stage when these MMAs finish
      }
      mma_commit_warp(smem_u32(&bar_acc));                   // accumulators complete
    }
  } else {
    // ------------------------------------------ converters, then the epilogue
    // 8 warps: thread ct converts row ct of the 256-row weight tile each stage.
    // Within each 8-k chunk the fp16 tile holds k in the order 0,4,1,5,2,6,3,7
    // (nibble pairs as they sit in a 32-bit word); the fp16 token copy is
    // written in the same order, so every 16-k MMA sums the same products.
    const int ct = threadIdx.x - 64;                         // 0..255
    const int n = n0 + ct;
    const bool row_ok = n < p.N;
    const int zrow = (p.ng + 1) / 2;
    const int stages_per_group = p.perch ? k_stages : p.G / kBK;
    const int ngroups = (k_stages + stages_per_group - 1) / stages_per_group;
    // The prefetched registers hold the loaded zero-point byte and scale bits
    // as they are; the nibble is picked and the scale doubled where they are
    // used, so no instruction waits for the load before then.  Per-channel
    // scales are applied in the epilogue.
    auto load_z = [&](int gi) -> uint32_t {
      if (p.sym || !row_ok || gi >= ngroups) return 0x88u;
      return __ldg(p.zeros + (size_t)n * zrow + gi / 2);
    };
    auto load_s = [&](int gi) -> uint32_t {
      if (p.perch || !row_ok || gi >= ngroups) return 0u;
      return __half_as_ushort(__ldg(p.scales + (size_t)n * p.ng + gi));
    };
    bool ok = true;
    auto convert = [&](int s, uint32_t zb, uint32_t sb) {      // s: this CTA's step (K step kb + s)
      const int slot = s % kStages;
      ok = __all_sync(0xffffffffu, ok && mbar_wait(smem_u32(&bar_full[slot]), (s / kStages) & 1, kWaitNs) &&
                                       !s_abort);
      if (ok) {
        const int gi = (kb + s) / stages_per_group;
        const uint32_t z = (gi & 1) ? (zb >> 4) : (zb & 15u);
        const uint32_t s2 = sb * 0x00010001u;                      // fp16x2 of the group scale
        const uint8_t* raw = raw_slot(slot) + ct * 32;
        uint8_t* wrow = w_slot(slot) + ct * 128;
        const uint32_t z_lo = f16x2_bias(z);                       // 1024 + z
        const uint32_t z_hi = (0x5400u | (z << 4)) * 0x00010001u;  // 64 + z
        const uint4 r0 = *reinterpret_cast<const uint4*>(raw);
        const uint4 r1 = *reinterpret_cast<const uint4*>(raw + 16);
        const uint32_t words[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
        for (int w = 0; w < 8; ++w) {
          const uint32_t a = words[w], b = words[w] >> 8;
          // (k0,k4), (k2,k6) as 1024 + u; (k1,k5), (k3,k7) as 64 + u (nibble in place,
          // one fp16 mantissa unit = 1/16 at 64); subtracting 1024 + z / 64 + z is exact
          uint32_t v0 = (a & 0x000F000Fu) | 0x64006400u, v1 = (a & 0x00F000F0u) | 0x54005400u;
          uint32_t v2 = (b & 0x000F000Fu) | 0x64006400u, v3 = (b & 0x00F000F0u) | 0x54005400u;
          v0 = f16x2_sub(v0, z_lo); v2 = f16x2_sub(v2, z_lo);
          v1 = f16x2_sub(v1, z_hi); v3 = f16x2_sub(v3, z_hi);
          if (!p.perch) {                                          // (u - z) s, one rounding
            v0 = f16x2_mul(v0, s2); v1 = f16x2_mul(v1, s2); v2 = f16x2_mul(v2, s2); v3 = f16x2_mul(v3, s2);
          }
          // 128-byte swizzle: 16-byte chunk c of row r lives at chunk c ^ (r & 7)
          *reinterpret_cast<uint4*>(wrow + ((w ^ (ct & 7)) << 4)) = make_uint4(v0, v1, v2, v3);
        }
      } else {
        give_up();
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bar_cvt[slot]));
    };
    // zero points and scales travel 4 groups ahead of their use in named
    // registers (slot = group mod 4, never indexed at run time)
    // (groups gb .. ge - 1 hold this CTA's K steps)
    const int gb = kb / stages_per_group, ge = (ke + stages_per_group - 1) / stages_per_group;
    uint32_t z0 = load_z(gb), z1 = load_z(gb + 1), z2 = load_z(gb + 2), z3 = load_z(gb + 3);
    uint32_t c0 = load_s(gb), c1 = load_s(gb + 1), c2 = load_s(gb + 2), c3 = load_s(gb + 3);
    auto group = [&](int gi, uint32_t& zs, uint32_t& cs) {
      const int s0 = std::max(gi * stages_per_group, kb), s1 = std::min((gi + 1) * stages_per_group, ke);
      for (int s = s0; s < s1; ++s) convert(s - kb, zs, cs);
      zs = load_z(gi + 4);
      cs = load_s(gi + 4);
    };
    for (int g0 = gb; g0 < ge; g0 += 4) {
      if (g0 + 0 < ge) group(g0 + 0, z0, c0);
      if (g0 + 1 < ge) group(g0 + 1, z1, c1);
      if (g0 + 2 < ge) group(g0 + 2, z2, c2);
      if (g0 + 3 < ge) group(g0 + 3, z3, c3);
    }

    // epilogue: TMEM lanes 32*(warp%4) .. +31 are this warp's rows (tokens);
    // warps 2-5 take output columns [0, 128), warps 6-9 columns [128, 256).
    // The fp16 token copy held x 2^-e (power-of-two token scaling): the main
    // term is multiplied by 2^e (loaded before the wait); a correction in its
    // own accumulator is unscaled, one in the main accumulators was scaled
    // with the tokens.
    float tsc0 = 1.0f, tsc1 = 1.0f;
    {
      const int tk = m0 + 32 * (warp & 3) + lane;
      if (tk < p.M) tsc0 = __ldg(p.tscale + tk);
      if (kMH > 1 && tk + 128 < p.M) tsc1 = __ldg(p.tscale + tk + 128);
    }
    ok = __all_sync(0xffffffffu, ok && mbar_wait(smem_u32(&bar_acc), 0, kWaitNs));
    if (!ok) give_up();
    tc_fence_after();
    if (!s_abort) {
      const int q = warp & 3;
      const int c_begin = ((warp - 2) >> 2) * (kBN / 2);
      // BM = 256: the second accumulator (columns 256..) holds tokens 128..255
      // and the correction is already in both
      const bool sep_comp = kMH == 1 && ncomp > 0;
#pragma unroll 1
      for (int it = 0; it < kMH * (kBN / 2 / 32); ++it) {
        const int mh = it / (kBN / 2 / 32), cch = c_begin / 32 + it % (kBN / 2 / 32);
        const int tok = m0 + 128 * mh + 32 * q + lane;
        uint32_t r[32], rc[32];
        tmem_ld_32cols(tmem + ((uint32_t)(32 * q) << 16) + mh * kBN + cch * 32, r);
        if (sep_comp) tmem_ld_32cols(tmem + ((uint32_t)(32 * q) << 16) + kBN + cch * 32, rc);
        tmem_ld_wait();
        const int n = n0 + cch * 32;
        if (n >= p.N) continue;
        float v[32];
        if (p.perch) {
          const uint4* sp = reinterpret_cast<const uint4*>(p.scales + n);   // per-channel: one scale per row
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint4 s8 = __ldg(sp + i);
            const uint32_t sw[4] = {s8.x, s8.y, s8.z, s8.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&sw[j]));
              v[8 * i + 2 * j] = __uint_as_float(r[8 * i + 2 * j]) * f.x;
              v[8 * i + 2 * j + 1] = __uint_as_float(r[8 * i + 2 * j + 1]) * f.y;
            }
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
        }
        const float tsc = mh ? tsc1 : tsc0;
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= tsc;
        if (sep_comp) {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] += __uint_as_float(rc[i]);
        }
        if (KS > 1) {
          // K split: this CTA's partial (scaled, with the correction on rank 0)
          // into its own shared memory; the cluster sums it below
          float* prow = reinterpret_cast<float*>(smem) + (32 * q + lane) * kRedStride + cch * 32;
#pragma unroll
          for (int i = 0; i < 8; ++i)
            reinterpret_cast<float4*>(prow)[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
          continue;
        }
        if (tok < p.M) {
          SPEAR_CHECK(&g_prefill_status, n + 32 <= p.N);
          if (p.out_f32) {
            float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.y) + (size_t)tok * p.N + n);
#pragma unroll
            for (int i = 0; i < 8; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.y) + (size_t)tok * p.N + n);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(pack_bf16x2(v[8 * i], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                                  pack_bf16x2(v[8 * i + 4], v[8 * i + 5]), pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
          }
        }
      }
    }
  }

  if (KS > 1) {
    // every thread of the cluster: rank R finishes output columns
    // [R 256 / KS, (R + 1) 256 / KS) of the tile, the partials summed in rank
    // order (16-byte shared-memory loads across the cluster, all in flight)
    cluster_sync();                                        // every partial is in place
    if (!s_abort) {
      const int c4n = kBN / KS / 4, cb = krank * (kBN / KS);
      const uint32_t red_base = smem_u32(smem);
      const bool f32 = p.out_f32 != 0;
      for (int idx = threadIdx.x; idx < BM * c4n; idx += kGemmThreads) {
        const int t = idx / c4n, col = cb + 4 * (idx % c4n);
        const int tok = m0 + t, n = n0 + col;
        const uint32_t la = red_base + (uint32_t)(t * kRedStride + col) * 4u;
        float4 pv[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (q < KS) pv[q] = dsmem_ld_f32x4(dsmem_addr(la, (uint32_t)q));
        float4 v = pv[0];
#pragma unroll
        for (int q = 1; q < 4; ++q)
          if (q < KS) { v.x += pv[q].x; v.y += pv[q].y; v.z += pv[q].z; v.w += pv[q].w; }
        if (tok >= p.M || n >= p.N) continue;               // N is a multiple of 64: n + 3 < N
        SPEAR_CHECK(&g_prefill_status, n + 4 <= p.N);
        const size_t o = (size_t)tok * p.N + n;
        if (f32) {
          *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.y) + o) = v;
        } else {
          *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.y) + o) =
              make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
        }
      }
    }
    cluster_sync();                                        // peers are done reading this CTA
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------- comp_down --
// One block = 32 tokens (4 token tiles of 8), all r+1 projection rows; 8 warps
// split K in 128-k chunks and are summed in a fixed order.  Same operand
// mapping as the decode producer: lane (g, c) owns 8 consecutive k per row.
constexpr int kCdThreads = 256;
constexpr int kCdWarps = kCdThreads / 32;
constexpr int kCdTok = 16;                    // tokens per cluster
constexpr int kCdMT = kCdTok / 8;
constexpr int kCdMaxCK = 8;                   // CTAs per cluster (K ranges)

struct CompDownParams {
  int M, K, r;
  int CK;               // cluster size: CTAs splitting K for one token tile
  const __nv_bfloat16* x;
  const __nv_bfloat16* A;
  const __nv_bfloat16* w_g;
  float b_g, alpha;
  int gh;               // vector-gate hidden width (0: the scalar gate)
  const float *gw1, *gc1, *gw2, *gc2;
  __nv_bfloat16* T2;    // [M][t2_cols]: T_hi in [0, r), T_lo in [r, 2r)
  int t2_cols;
  __half* x16;          // optional [M][K] fp16 copy of x for the GEMM (NULL: not written)
  float* tscale;        // with x16: [M] the scale 2^e_m of each token's copy (written here)
  int scale_T;          // T2 holds T_m 2^-e_m (the correction joins the GEMM's scaled accumulators)
};

// 8 consecutive bf16 (k0..k7), times the token's scale 2^-e (a power of two,
// so exact), -> 8 fp16 in the GEMM's operand order within an 8-k chunk:
// (k0,k4) (k1,k5) (k2,k6) (k3,k7).
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v, float sc) {
  const float x0 = bf16x2_lo(v.x) * sc, x1 = bf16x2_hi(v.x) * sc, x2 = bf16x2_lo(v.y) * sc, x3 = bf16x2_hi(v.y) * sc;
  const float x4 = bf16x2_lo(v.z) * sc, x5 = bf16x2_hi(v.z) * sc, x6 = bf16x2_lo(v.w) * sc, x7 = bf16x2_hi(v.w) * sc;
  auto h2 = [](float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  };
  return make_uint4(h2(x0, x4), h2(x1, x5), h2(x2, x6), h2(x3, x7));
}

// One cluster of CK CTAs per 16-token tile; CTA `rank` covers the 32-k pieces
// [rank n / CK, (rank + 1) n / CK) of K (and writes the fp16 token copy of
// that range).  Its 8 warps take interleaved pieces, U at a time with every
// load in flight; the warp partials are summed in warp order, the CK partials
// in rank order through distributed shared memory, then rank 0 forms the gate
// and T = alpha g (A x) as bf16 hi + lo.
template <int RT>
__global__ void __launch_bounds__(kCdThreads) comp_down_kernel(const CompDownParams p) {
  constexpr int U = RT <= 3 ? 2 : 1;                       // pieces in flight per warp
  __shared__ float red[kCdWarps][kCdMT][4][32];
  __shared__ float part[RT * 16][kCdTok];                  // [projection row][token]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int CK = p.CK;
  const int rank = (int)cluster_ctarank();
  const int tok0 = (int)(blockIdx.x / CK) * kCdTok;
  const int npieces = p.K / 32;
  const int pc0 = rank * npieces / CK, pc1 = (rank + 1) * npieces / CK;
  // Power-of-two token scaling of the fp16 copy: the copy is written
  // unscaled while each thread keeps the max |x| of its tokens (bits of a
  // non-negative float order like the values; NaN above inf); the cluster's
  // maxima meet in distributed shared memory with the partials, and only a
  // token whose max reaches 2^15 (rare) is converted again, scaled.
  __shared__ unsigned s_wmax[kCdWarps][kCdTok];            // per warp
  __shared__ unsigned s_tmax[kCdTok];                      // this CTA's K range
  __shared__ float s_tsc[kCdTok];                          // 2^-e of each token of the tile
  __shared__ int s_tany;                                   // some token of the tile is scaled
  if (threadIdx.x == 0) s_tany = 0;                        // read after two cluster barriers
  unsigned tm[kCdMT];
#pragma unroll
  for (int t = 0; t < kCdMT; ++t) tm[t] = 0u;
  // the vector gate's weights (h <= 32, r <= 64), copied by rank 0 while its
  // K slice streams
  __shared__ __align__(16) float gate_s[gate_smem_floats(64, 32)];
  if (rank == 0 && p.gh > 0)
    stage_gate_weights_async(p.gw1, p.gw2, p.gc1, p.gc2, p.r, p.gh, gate_s, threadIdx.x, kCdThreads);
  float acc[RT][kCdMT][4];
#pragma unroll
  for (int rt = 0; rt < RT; ++rt)
#pragma unroll
    for (int t = 0; t < kCdMT; ++t)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[rt][t][i] = 0.0f;
  for (int pb = pc0 + warp; pb < pc1; pb += U * kCdWarps) {
    uint4 xv[U][kCdMT], va[U][RT], vb[U][RT];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int pc = pb + u * kCdWarps;
      const bool ok = pc < pc1;
      const int kb = pc * 32 + 8 * c;
#pragma unroll
      for (int t = 0; t < kCdMT; ++t) {
        const int tok = tok0 + t * 8 + g;
        xv[u][t] = (ok && tok < p.M) ? ldg16(p.x + (size_t)tok * p.K + kb) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int rt = 0; rt < RT; ++rt) {
        const int rlo = rt * 16 + g, rhi = rlo + 8;
        // (row r is w_g . x for the scalar gate; with the vector gate w_g may be NULL)
        va[u][rt] = !ok ? make_uint4(0, 0, 0, 0)
                        : rlo < p.r ? ldg16(p.A + (size_t)rlo * p.K + kb)
                                    : (rlo == p.r && p.w_g) ? ldg16(p.w_g + kb) : make_uint4(0, 0, 0, 0);
        vb[u][rt] = !ok ? make_uint4(0, 0, 0, 0)
                        : rhi < p.r ? ldg16(p.A + (size_t)rhi * p.K + kb)
                                    : (rhi == p.r && p.w_g) ? ldg16(p.w_g + kb) : make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int pc = pb + u * kCdWarps;
      if (p.x16 && pc < pc1) {
        const int kb = pc * 32 + 8 * c;
#pragma unroll
        for (int t = 0; t < kCdMT; ++t) {
          const int tok = tok0 + t * 8 + g;
          tm[t] = max(tm[t], __float_as_uint(bf16x8_absmax(xv[u][t])));   // zeros past M
          if (tok < p.M) *reinterpret_cast<uint4*>(p.x16 + (size_t)tok * p.K + kb) = bf16x8_to_f16x8(xv[u][t], 1.0f);
        }
      }
#pragma unroll
      for (int rt = 0; rt < RT; ++rt)
#pragma unroll
        for (int t = 0; t < kCdMT; ++t) {
          mma_bf16_16816(acc[rt][t], va[u][rt].x, vb[u][rt].x, va[u][rt].y, vb[u][rt].y, xv[u][t].x, xv[u][t].y);
          mma_bf16_16816(acc[rt][t], va[u][rt].z, vb[u][rt].z, va[u][rt].w, vb[u][rt].w, xv[u][t].z, xv[u][t].w);
        }
    }
  }
  if (p.x16) {
    // lanes 4g .. 4g + 3 hold tokens g and 8 + g of the tile
#pragma unroll
    for (int t = 0; t < kCdMT; ++t) {
      tm[t] = max(tm[t], __shfl_xor_sync(0xffffffffu, tm[t], 1));
      tm[t] = max(tm[t], __shfl_xor_sync(0xffffffffu, tm[t], 2));
      if (c == 0) s_wmax[warp][t * 8 + g] = tm[t];
    }
  }
  // fixed-order sum over the warps, one projection-row tile at a time
#pragma unroll
  for (int rt = 0; rt < RT; ++rt) {
#pragma unroll
    for (int t = 0; t < kCdMT; ++t)
#pragma unroll
      for (int i = 0; i < 4; ++i) red[warp][t][i][lane] = acc[rt][t][i];
    __syncthreads();
    for (int e = threadIdx.x; e < kCdMT * 4 * 32; e += kCdThreads) {
      const int t = e / 128, i = (e / 32) & 3, ln = e & 31;
      float s = 0.0f;
#pragma unroll
      for (int w = 0; w < kCdWarps; ++w) s += red[w][t][i][ln];
      // C fragment element i of lane ln: row (ln/4) + 8 (i/2), token 2 (ln%4) + (i%2)
      part[rt * 16 + (ln >> 2) + 8 * (i >> 1)][t * 8 + 2 * (ln & 3) + (i & 1)] = s;
    }
    __syncthreads();
  }
  if (p.x16 && threadIdx.x < kCdTok) {                     // (the warps' maxima are behind the barriers above)
    unsigned m = 0u;
#pragma unroll
    for (int w = 0; w < kCdWarps; ++w) m = max(m, s_wmax[w][threadIdx.x]);
    s_tmax[threadIdx.x] = m;
  }
  cluster_sync();                                          // every CTA's partial and maxima are in place
  if (p.x16 && threadIdx.x < kCdTok) {
    unsigned m = 0u;
    for (int q = 0; q < CK; ++q)
      m = max(m, __float_as_uint(dsmem_ld_f32(dsmem_addr(smem_u32(&s_tmax[threadIdx.x]), (uint32_t)q))));
    const int ex = token_scale_exp(__uint_as_float(m));
    s_tsc[threadIdx.x] = exp2_int(-ex);
    if (ex > 0) s_tany = 1;
    const int tok = tok0 + (int)threadIdx.x;
    if (rank == 0 && tok < p.M) {
      p.tscale[tok] = exp2_int(ex);
      if (m > 0x7f7fffffu) record_status(&g_prefill_status, DEV_ERR_INVALID);   // inf or NaN
    }
  }
  if (rank == 0) {
    // the CK partials in rank order (all loads in flight), into this CTA's own
    // partial; then row r is the gate logit, rows 0..r-1 the down-projection
    for (int e = threadIdx.x; e < (p.r + 1) * kCdTok; e += kCdThreads) {
      const uint32_t la = smem_u32(&part[0][0] + e);
      float pv[kCdMaxCK];
#pragma unroll
      for (int q = 0; q < kCdMaxCK; ++q)
        if (q < CK) pv[q] = dsmem_ld_f32(dsmem_addr(la, (uint32_t)q));
      float v = 0.0f;
#pragma unroll
      for (int q = 0; q < kCdMaxCK; ++q)
        if (q < CK) v += pv[q];
      (&part[0][0])[e] = v;
    }
  }
  cluster_sync();                                          // peers are done reading; rank 0's sums in place
  if (p.x16 && s_tany) {
    // rare: the tokens that take a scale, converted again over this CTA's K range
    const int units = (pc1 - pc0) * 4;                     // 8-k units
    for (int e = threadIdx.x; e < kCdTok * units; e += kCdThreads) {
      const int t = e / units, tok = tok0 + t;
      if (tok < p.M && s_tsc[t] != 1.0f) {
        const size_t o = (size_t)tok * p.K + pc0 * 32 + (e % units) * 8;
        *reinterpret_cast<uint4*>(p.x16 + o) = bf16x8_to_f16x8(ldg16(p.x + o), s_tsc[t]);
      }
    }
  }
  __shared__ float hid[kCdTok * gate_hid_stride(32)];      // [16 tokens][h | 1]
  if (rank == 0 && p.gh > 0) {
    // vector gate on the summed partial (part[j][m]): t scaled in place by gamma(t)
    const GateSmem gt(gate_s, p.r, p.gh);
    cp_async_wait<0>();
    __syncthreads();
    vector_gate_hidden(&part[0][0], 1, kCdTok, kCdTok, gt, hid, threadIdx.x, kCdThreads);
    __syncthreads();
    vector_gate_apply(&part[0][0], 1, kCdTok, kCdTok, gt, hid, threadIdx.x, kCdThreads);
    __syncthreads();
  }
  if (rank == 0) {
    for (int e = threadIdx.x; e < kCdTok * p.r; e += kCdThreads) {
      const int m = e / p.r, j = e % p.r;
      const int tok = tok0 + m;
      const float gate = p.gh > 0 ? 1.0f : 1.0f / (1.0f + expf(-(part[p.r][m] + p.b_g)));
      // T_m 2^-e_m when the correction joins the GEMM's scaled accumulators
      const float tv = p.alpha * gate * part[j][m] * (p.scale_T ? s_tsc[m] : 1.0f);
      const __nv_bfloat16 hi = __float2bfloat16_rn(tv);
      const __nv_bfloat16 lo = __float2bfloat16_rn(tv - __bfloat162float(hi));
      if (tok < p.M) {
        p.T2[(size_t)tok * p.t2_cols + j] = hi;
        p.T2[(size_t)tok * p.t2_cols + p.r + j] = lo;
      }
    }
  }
}

// --------------------------------------------------------------- to_fp16 --
// fp16 copy of the activations for the GEMM when no compensator pass reads
// them, one token row per block at a time: the row's 16-byte units are loaded
// into registers (CPT per thread) while the row's max |x| is taken, then
// written with the row's power-of-two scale 2^-e (e = 0 unless the max reaches
// 2^15).  CPT = 0: rows longer than 4096 units, read twice.
template <int CPT>
__global__ void __launch_bounds__(256) to_fp16_kernel(const uint4* __restrict__ x, uint4* __restrict__ x16,
                                                      float* __restrict__ tscale, int M, int K) {
  constexpr int kT = 256;
  __shared__ unsigned s_max[2][kT / 32];                   // per warp, alternating rows
  const int k8 = K / 8, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int par = 0;
  for (int m = blockIdx.x; m < M; m += gridDim.x, par ^= 1) {
    const uint4* row = x + (size_t)m * k8;
    uint4* out = x16 + (size_t)m * k8;
    constexpr int kR = CPT > 0 ? CPT : 1;
    uint4 v[kR];
    unsigned am = 0u;                                      // bits of max |x| (NaN above inf)
    if constexpr (CPT > 0) {
#pragma unroll
      for (int i = 0; i < CPT; ++i) {
        const int j = (int)threadIdx.x + kT * i;
        v[i] = j < k8 ? __ldg(row + j) : make_uint4(0, 0, 0, 0);
        am = max(am, __float_as_uint(bf16x8_absmax(v[i])));
      }
    } else {
      for (int j = threadIdx.x; j < k8; j += kT) am = max(am, __float_as_uint(bf16x8_absmax(__ldg(row + j))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am = max(am, __shfl_xor_sync(0xffffffffu, am, o));
    if (lane == 0) s_max[par][warp] = am;
    __syncthreads();                                       // (the other slot is still being read for the last row)
    unsigned mx = 0u;
#pragma unroll
    for (int w = 0; w < kT / 32; ++w) mx = max(mx, s_max[par][w]);
    const int ex = token_scale_exp(__uint_as_float(mx));
    const float sc = exp2_int(-ex);
    if constexpr (CPT > 0) {
#pragma unroll
      for (int i = 0; i < CPT; ++i) {
        const int j = (int)threadIdx.x + kT * i;
        if (j < k8) out[j] = bf16x8_to_f16x8(v[i], sc);
      }
    } else {
      for (int j = threadIdx.x; j < k8; j += kT) out[j] = bf16x8_to_f16x8(__ldg(row + j), sc);
    }
    if (threadIdx.x == 0) {
      tscale[m] = exp2_int(ex);
      if (mx > 0x7f7fffffu) record_status(&g_prefill_status, DEV_ERR_INVALID);   // inf or NaN
    }
  }
}

// ----------------------------------------------------------- comp_up_add --
// Y[m][n] = Y32[m][n] + sum_j (T_hi + T_lo)[m][j] B[n][j], rounded once.
// One warp = 16 tokens x 64 outputs (8 mma n-tiles), A operand = T rows,
// B operand = rows of B.  Y32 is the plain GEMM's fp32 result (it may be y
// itself when y is fp32).
struct CompUpParams {
  int M, N, r, t2_cols, out_f32;
  const __nv_bfloat16* T2;
  const __nv_bfloat16* B;
  const float* y32;
  void* y;
};

__global__ void __launch_bounds__(256) comp_up_add_kernel(const CompUpParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int tok0 = (blockIdx.y * 8 + warp) * 16;
  const int nb = blockIdx.x * 64;
  if (tok0 >= p.M) return;
  float acc[8][4];
#pragma unroll
  for (int t = 0; t < 8; ++t)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[t][i] = 0.0f;
  const int tlo = min(tok0 + g, p.M - 1), thi = min(tok0 + g + 8, p.M - 1);
  for (int part = 0; part < 2; ++part) {                     // T_hi, then T_lo
    for (int j0 = 0; j0 < p.r; j0 += 16) {
      const uint32_t* Tl = reinterpret_cast<const uint32_t*>(p.T2 + (size_t)tlo * p.t2_cols + part * p.r + j0);
      const uint32_t* Th = reinterpret_cast<const uint32_t*>(p.T2 + (size_t)thi * p.t2_cols + part * p.r + j0);
      const uint32_t a0 = Tl[c], a1 = Th[c], a2 = Tl[c + 4], a3 = Th[c + 4];
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const uint32_t* Bn = reinterpret_cast<const uint32_t*>(p.B + (size_t)(nb + t * 8 + g) * p.r + j0);
        mma_bf16_16816(acc[t], a0, a1, a2, a3, __ldg(Bn + c), __ldg(Bn + c + 4));
      }
    }
  }
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    const int n = nb + t * 8 + 2 * c;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int tok = tok0 + g + 8 * hh;
      if (tok >= p.M) continue;
      SPEAR_CHECK(&g_prefill_status, n + 2 <= p.N);
      const float2 m32 = *reinterpret_cast<const float2*>(p.y32 + (size_t)tok * p.N + n);
      const float v0 = m32.x + acc[t][2 * hh], v1 = m32.y + acc[t][2 * hh + 1];
      if (p.out_f32) {
        *reinterpret_cast<float2*>(reinterpret_cast<float*>(p.y) + (size_t)tok * p.N + n) = make_float2(v0, v1);
      } else {
        *reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<__nv_bfloat16*>(p.y) + (size_t)tok * p.N + n) =
            __floats2bfloat162_rn(v0, v1);
      }
    }
  }
}

// ----------------------------------------------------------------- host --

int t2_cols_for(int r) { return 2 * r; }
size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// AUTO takes the fused mode: with the clustered down-projection it is the
// faster one at every measured shape (4-14 % over the plain W4 GEMM).
int resolve_mode(int mode) { return mode == SPEAR_PREFILL_AUTO ? SPEAR_PREFILL_FUSED : mode; }

// x16: fp16 copy of the activations [M][K].
// Tile height: 256 tokens (two M = 128 MMAs on each converted weight tile)
// where it takes fewer time units than 128-token tiles.  One CTA per SM; a
// 256-token tile's K loop takes ~1.35x as long as a 128-token one's (measured
// stage times on GB300), so cost = waves x (1 or 1.35).  Per-channel scales
// multiply the accumulator in the epilogue, so with a fused correction (its
// own accumulator) tiles stay at 128 tokens.
int pick_bm(int M, int N, bool perch_fused, int num_sms) {
  if (perch_fused) return 128;
  const long long ntiles = (N + kBN - 1) / kBN;
  const long long w128 = (ntiles * ((M + 127) / 128) + num_sms - 1) / num_sms;
  const long long w256 = (ntiles * ((M + 255) / 256) + num_sms - 1) / num_sms;
  return 135 * w256 < 100 * w128 ? 256 : 128;
}

// K split for grids that would leave most SMs idle (a few 128-token tiles:
// each CTA would dequantise a whole 256-row slab of the weight alone): up to
// 4 CTAs of a cluster take equal K ranges while the grid stays within one wave.
int pick_ks(int BM, int ctas, int k_steps, int num_sms) {
  int ks = 1;
  if (BM != 128) return ks;
  while (ks < 4 && 2 * ks * ctas <= num_sms && k_steps >= 16 * ks) ks *= 2;
  return ks;
}

int launch_gemm(const spear_w4_layer& L, const __half* x16, const float* tscale, int M, void* y, int out_f32,
                const __nv_bfloat16* T2, int r_fused, cudaStream_t st) {
  DeviceInfo di;
  if (int rc = device_info(&di)) return rc;
  const bool perch = L.group_size == L.K;
  const int BM = pick_bm(M, L.N, perch && r_fused > 0, di.num_sms);
  if (log_plans())
    fprintf(stderr, "[spear] prefill gemm N=%d K=%d M=%d G=%d fused_rank=%d: %d-token tiles\n", L.N, L.K, M,
            L.group_size, r_fused, BM);
  CUtensorMap tm_x, tm_wq, tm_t, tm_b;
  if (int rc = make_tmap(&tm_x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, x16, L.K, M, kBK, BM,
                         CU_TENSOR_MAP_SWIZZLE_128B)) return rc;
  if (int rc = make_tmap(&tm_wq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, L.qweight, L.K / 2, L.N, kBK / 2, kBN,
                         CU_TENSOR_MAP_SWIZZLE_NONE)) return rc;
  GemmParams p{};
  p.M = M; p.N = L.N; p.K = L.K; p.G = L.group_size; p.ng = L.K / L.group_size; p.sym = L.symmetric;
  p.perch = L.group_size == L.K;
  p.scales = reinterpret_cast<const __half*>(L.scales);
  p.zeros = L.zeros;
  p.y = y; p.out_f32 = out_f32;
  p.tscale = tscale;
  p.r = r_fused;
  if (r_fused > 0) {
    const int tcols = t2_cols_for(r_fused);
    const int tbox = std::min(tcols, 64);
    p.t_row_bytes = tbox * 2;
    p.b_row_bytes = r_fused * 2;
    p.comp_stages = (2 * r_fused + 63) / 64;
    if (int rc = make_tmap(&tm_t, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T2, tcols, M, tbox, BM,
                           swizzle_for(p.t_row_bytes))) return rc;
    if (int rc = make_tmap(&tm_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, L.B, r_fused, L.N, r_fused, kBN,
                           swizzle_for(p.b_row_bytes))) return rc;
  } else {
    tm_t = tm_x;
    tm_b = tm_x;
  }
  auto fn = BM == 256 ? w4_gemm_tc<256> : w4_gemm_tc<128>;
  const size_t smem = BM == 256 ? (size_t)TileCfg<256>::kStages * TileCfg<256>::kStageBytes + 1024
                                : (size_t)TileCfg<128>::kStages * TileCfg<128>::kStageBytes + 1024;
  static_assert((size_t)128 * kRedStride * 4 <= (size_t)TileCfg<128>::kStages * TileCfg<128>::kStageBytes,
                "the K-split partial fits in the 128-token tile's stage buffers");
  if (int rc = ensure_smem_limit(reinterpret_cast<const void*>(fn), smem)) return rc;
  dim3 grid((L.N + kBN - 1) / kBN, (M + BM - 1) / BM);
  if (grid.y > 65535) return fail(SPEAR_ERR_UNSUPPORTED, "prefill: M=%d too large", M);
  p.ks = pick_ks(BM, (int)(grid.x * grid.y), L.K / kBK, di.num_sms);
  if (log_plans() && p.ks > 1) fprintf(stderr, "[spear] prefill gemm: K split over %d CTAs\n", p.ks);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid.x, grid.y, p.ks);
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = p.ks;
  cfg.attrs = attr;
  cfg.numAttrs = p.ks > 1 ? 1 : 0;
  return cuda_check(cudaLaunchKernelEx(&cfg, fn, tm_x, tm_wq, tm_t, tm_b, p), "prefill gemm launch");
}

int launch_comp_down(const spear_w4_layer& L, const uint16_t* x, int M, __nv_bfloat16* T2, __half* x16,
                     float* tscale, int scale_T, cudaStream_t st) {
  DeviceInfo di;
  if (int rc = device_info(&di)) return rc;
  CompDownParams p{};
  p.x16 = x16;
  p.tscale = tscale;
  p.scale_T = scale_T;
  p.M = M; p.K = L.K; p.r = L.rank;
  p.x = reinterpret_cast<const __nv_bfloat16*>(x);
  p.A = reinterpret_cast<const __nv_bfloat16*>(L.A);
  p.w_g = reinterpret_cast<const __nv_bfloat16*>(L.w_g);
  p.b_g = L.b_g; p.alpha = L.alpha;
  p.gh = L.gate_hidden; p.gw1 = L.gate_w1; p.gc1 = L.gate_c1; p.gw2 = L.gate_w2; p.gc2 = L.gate_c2;
  p.T2 = T2; p.t2_cols = t2_cols_for(L.rank);
  // K ranges per token tile: as many as keep the grid within two CTAs per SM
  // (rounded down: 2048 tokens on 152 SMs take 2 ranges, 256 CTAs, 67 us for
  // 4096 x 4096 against 73 us with 3 ranges, 384 CTAs; 512 tokens take 8)
  const int tiles = (M + kCdTok - 1) / kCdTok;
  p.CK = std::max(1, std::min(kCdMaxCK, (2 * di.num_sms) / tiles));
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(tiles * p.CK));
  cfg.blockDim = dim3(kCdThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)p.CK;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaError_t e;
  switch ((L.rank + 1 + 15) / 16) {
    case 2: e = cudaLaunchKernelEx(&cfg, comp_down_kernel<2>, p); break;
    case 3: e = cudaLaunchKernelEx(&cfg, comp_down_kernel<3>, p); break;
    default: e = cudaLaunchKernelEx(&cfg, comp_down_kernel<5>, p); break;
  }
  return cuda_check(e, "comp_down launch");
}

int launch_to_fp16(const uint16_t* x, __half* x16, float* tscale, int M, int K, cudaStream_t st) {
  DeviceInfo di;
  if (int rc = device_info(&di)) return rc;
  // K % 128 == 0, so every row is a whole number of 16-byte units
  const int units = K / 8;
  auto fn = units <= 256 ? to_fp16_kernel<1> : units <= 512 ? to_fp16_kernel<2> : units <= 1024 ? to_fp16_kernel<4>
          : units <= 2048 ? to_fp16_kernel<8> : units <= 4096 ? to_fp16_kernel<16> : to_fp16_kernel<0>;
  const unsigned blocks = (unsigned)std::min(M, di.num_sms * 8);
  fn<<<blocks, 256, 0, st>>>(reinterpret_cast<const uint4*>(x), reinterpret_cast<uint4*>(x16), tscale, M, K);
  return cuda_check(cudaGetLastError(), "to_fp16 launch");
}

int launch_comp_up(const spear_w4_layer& L, int M, void* y, int out_f32, const float* y32, const __nv_bfloat16* T2,
                   cudaStream_t st) {
  CompUpParams p{};
  p.M = M; p.N = L.N; p.r = L.rank; p.t2_cols = t2_cols_for(L.rank); p.out_f32 = out_f32;
  p.T2 = T2;
  p.y32 = y32;
  p.B = reinterpret_cast<const __nv_bfloat16*>(L.B);
  p.y = y;
  dim3 grid(L.N / 64, (M + 127) / 128);
  comp_up_add_kernel<<<grid, 256, 0, st>>>(p);
  return cuda_check(cudaGetLastError(), "comp_up launch");
}

struct StreamEvents {
  cudaEvent_t fork = nullptr, join = nullptr;
};

int stream_events(StreamEvents* ev) {
  static std::mutex mu;
  static StreamEvents cache[64];
  static bool made[64] = {};
  int dev = 0;
  if (int rc = cuda_check(cudaGetDevice(&dev), "cudaGetDevice")) return rc;
  if (dev < 0 || dev >= 64) return fail(SPEAR_ERR_UNSUPPORTED, "device index %d", dev);
  std::lock_guard<std::mutex> lk(mu);
  if (!made[dev]) {
    if (int rc = cuda_check(cudaEventCreateWithFlags(&cache[dev].fork, cudaEventDisableTiming), "event")) return rc;
    if (int rc = cuda_check(cudaEventCreateWithFlags(&cache[dev].join, cudaEventDisableTiming), "event")) return rc;
    made[dev] = true;
  }
  *ev = cache[dev];
  return SPEAR_OK;
}

// Workspace: [T2: M x 2r bf16][X16: M x K fp16][token scales: M fp32]
// [Y32: M x N fp32, stream mode with bf16 output only]
struct WsLayout {
  size_t t2, x16, ts, y32, total;
};

WsLayout ws_layout(const spear_w4_layer& L, int M, int mode, int out_f32) {
  const bool comp = L.comp_enabled && L.rank > 0;
  WsLayout w{};
  size_t off = 0;
  w.t2 = off;  off = align256(off + (comp ? (size_t)M * t2_cols_for(L.rank) * 2 : 0));
  w.x16 = off; off = align256(off + (size_t)M * L.K * 2);
  w.ts = off;  off = align256(off + (size_t)M * 4);
  w.y32 = off;
  if (comp && resolve_mode(mode) == SPEAR_PREFILL_STREAM && !out_f32) off = align256(off + (size_t)M * L.N * 4);
  w.total = off;
  return w;
}

}  // namespace

int prefill_workspace_bytes(const spear_w4_layer& L, int M, int mode, size_t* bytes) {
  *bytes = ws_layout(L, M, mode, 0).total;          // the bf16-output size covers fp32 output too
  return SPEAR_OK;
}

int launch_prefill(const spear_w4_layer& L, const uint16_t* x, int M, void* y, int out_f32, int mode, void* ws,
                   size_t ws_bytes, cudaStream_t st, cudaStream_t st_aux) {
  DeviceInfo di;
  if (int rc = device_info(&di)) return rc;
  const bool comp = L.comp_enabled && L.rank > 0;
  const WsLayout lay = ws_layout(L, M, mode, out_f32);
  if (!ws || ws_bytes < lay.total)
    return fail(SPEAR_ERR_WORKSPACE, "prefill: workspace of %zu B is smaller than the %zu B needed", ws_bytes,
                lay.total);
  if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0)
    return fail(SPEAR_ERR_INVALID_ARG, "prefill: workspace must be 256-byte aligned");
  char* base = reinterpret_cast<char*>(ws);
  __nv_bfloat16* T2 = reinterpret_cast<__nv_bfloat16*>(base + lay.t2);
  __half* x16 = reinterpret_cast<__half*>(base + lay.x16);
  float* ts = reinterpret_cast<float*>(base + lay.ts);
  if (!comp) {
    if (int rc = launch_to_fp16(x, x16, ts, M, L.K, st)) return rc;
    return launch_gemm(L, x16, ts, M, y, out_f32, nullptr, 0, st);
  }
  if (resolve_mode(mode) == SPEAR_PREFILL_FUSED) {
    // 256-token tiles add the correction into the main (token-scaled) accumulators
    const bool perch = L.group_size == L.K;
    const int scale_T = pick_bm(M, L.N, perch, di.num_sms) == 256 ? 1 : 0;
    if (int rc = launch_comp_down(L, x, M, T2, x16, ts, scale_T, st)) return rc;
    return launch_gemm(L, x16, ts, M, y, out_f32, T2, L.rank, st);
  }
  // stream mode: the down-projection runs on st_aux beside the W4 GEMM on st;
  // the GEMM writes fp32 so the up-projection-and-add rounds only once
  if (!st_aux || st_aux == st) return fail(SPEAR_ERR_INVALID_ARG, "prefill: stream mode needs a distinct stream_aux");
  float* y32 = out_f32 ? reinterpret_cast<float*>(y) : reinterpret_cast<float*>(base + lay.y32);
  StreamEvents ev;
  if (int rc = stream_events(&ev)) return rc;
  if (int rc = cuda_check(cudaEventRecord(ev.fork, st), "fork record")) return rc;
  if (int rc = cuda_check(cudaStreamWaitEvent(st_aux, ev.fork, 0), "fork wait")) return rc;
  if (int rc = launch_comp_down(L, x, M, T2, nullptr, nullptr, 0, st_aux)) return rc;
  if (int rc = cuda_check(cudaEventRecord(ev.join, st_aux), "join record")) return rc;
  if (int rc = launch_to_fp16(x, x16, ts, M, L.K, st)) return rc;
  if (int rc = launch_gemm(L, x16, ts, M, y32, 1, nullptr, 0, st)) return rc;
  if (int rc = cuda_check(cudaStreamWaitEvent(st, ev.join, 0), "join wait")) return rc;
  return launch_comp_up(L, M, y, out_f32, y32, T2, st);
}

int read_and_clear_status_prefill(unsigned* out, cudaStream_t st) {
  void* addr = nullptr;
  if (int rc = cuda_check(cudaGetSymbolAddress(&addr, g_prefill_status), "prefill status address")) return rc;
  if (int rc = cuda_check(cudaMemcpyAsync(out, addr, sizeof(unsigned), cudaMemcpyDeviceToHost, st), "read prefill status")) return rc;
  if (int rc = cuda_check(cudaStreamSynchronize(st), "read prefill status")) return rc;
  return cuda_check(cudaMemsetAsync(addr, 0, sizeof(unsigned), st), "clear prefill status");
}

}  // namespace spear
