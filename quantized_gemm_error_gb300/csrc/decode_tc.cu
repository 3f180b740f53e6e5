// decode_tc.cu -- decode path of the gated W4 + low-rank compensated linear on
// the 5th-generation tensor cores, one launch per layer (SPEAR explainer,
// Technical Summary 2.2 A: in the memory-bound decode phase the compensator
// runs inside the low-bit GEMM's launch).  Serves the larger token counts
// (17..64), where the per-weight arithmetic outgrows the warp-level MMAs of
// decode.cu, and the wide layers whose warp-level plan does not fit.
//
//   y[m][n] = sum_k (u[n][k] - z[n][g]) s[n][g] x[m][k]  +  sum_j B[n][j] T[m][j]
//   T[m][j] = alpha g_m (A x_m)[j],   g_m = sigmoid(w_g . x_m + b_g)
//
// Work split.  The weight is cut into 256-row tiles; each tile belongs to one
// thread-block cluster of S CTAs (one per SM) that split its K range in
// 256-k units (rank j takes units j, j + S, ...), so a tile's partial sums
// meet in distributed shared memory and never touch HBM.  Before the tile
// clusters come RT small "producer" clusters, one per 16-row tile of
// [A; w_g], that compute P = [A; w_g] x (rank r + 1 rows) over K slices with
// mma.sync and publish it through the workspace; the last of them to publish
// forms T from P (either gate) and publishes it too, and the tile CTAs read
// T only in their epilogue.
//
// Tile CTA (704 threads):
//   warp 20   TMA: raw int4 units (256 rows x 128 bytes, 128-byte swizzle) and
//             token tiles x[0:NP][k:k+64] (bf16), each into its own ring;
//   warps 4-19 turn each 64-k step of int4 codes into (u - z) s in fp16 (one
//             rounding; the nibble enters as the mantissa of 1024 or 64, so
//             the subtraction of 1024 + z or 64 + z is exact), written in the
//             tensor core's swizzled K-major layout; after the last MMA they
//             drain the accumulator into this CTA's partial in shared memory;
//   warps 0-3 convert the token tile to fp16 (exact for |x| < 65504) and
//             flag the tokens holding a larger value, then read the published
//             T hi/lo that the last producer CTA formed (tc_form_T: either
//             gate) into the spent ring; after the drain the converter warps
//             recompute a flagged token's partial in fp32 (tc_exact_rows);
//   warp 21   one thread issues tcgen05.mma with the tokens as the 64-row A
//             operand and the weights as the 256-column B operand:
//             D[64 x 256] (+)= X[64 x 16] W[256 x 16]^T, fp32 in tensor memory.
// Epilogue: warps 0-19 add B T into the partial rows this CTA finishes; then
// the S partials of the cluster are summed in a fixed order through DSMEM,
// each CTA finishing 256 / S rows of y.
//
// Shared memory carries every weight several times (int4 in, fp16 out, fp16
// read by the tensor core: ~10 bytes per int4 byte), which bounds this kernel
// near a quarter of what an SM draws from HBM; decode.cu's register path does
// not have that cost and serves M <= 16.
#include <cuda.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"
#include "tmap.h"

namespace spear {
namespace {

__device__ unsigned g_dtc_status;

using namespace sm100;

constexpr int kTileRows = 256;                  // weight rows per tile CTA (MMA N)
constexpr int kStepK = 64;                      // k per MMA step: one 128-byte row of fp16
constexpr int kUnitK = 256;                     // k per raw int4 unit: 128 bytes per row
constexpr int kRawBytes = kTileRows * kUnitK / 2;   // 32 KB
constexpr int kBfBytes = kTileRows * kStepK * 2;    // 32 KB of fp16 weights per step
constexpr int kX16Bytes = 64 * kStepK * 2;          // 8 KB: 64 token rows (MMA M = 64)
constexpr int kRawStages = 2, kXrStages = 2, kX16Stages = 3, kMaxBfStages = 3;
constexpr int kRedStride = kTileRows + 4;       // floats per token row of the partial (16-byte rows)
constexpr int kXWarps = 4;                      // warps 0-3: token conversion, TMEM drain
constexpr int kConvWarp0 = 4, kConvWarps = 16;  // warps 4-19: weight conversion (two threads per row)
constexpr int kTmaWarp = 20, kMmaWarp = 21;
constexpr int kThreads = 704;
constexpr int kMaxS = 8;
constexpr uint64_t kPipeWaitNs = 2000ull * 1000 * 1000;   // 2 s: far beyond any legitimate wait
constexpr uint64_t kTWaitNs = 200ull * 1000 * 1000;       // 200 ms for the published T

struct TcParams {
  int N, K, M, ng, sym;
  const uint8_t* qweight;
  int S;                    // CTAs per cluster
  int RT;                   // producer clusters, one per 16-row tile of [A; w_g] (0: none)
  int units;                // 256-k units of K
  int bf_stages;             // fp16 weight steps in flight (2 or 3)
  int r;                    // rank (0 when the compensator is off)
  int n_consumers;          // tile CTAs (they read P)
  const __half* scales;
  const uint8_t* zeros;
  const __nv_bfloat16* x;
  void* y;
  int out_f32;
  const __nv_bfloat16* A;
  const __nv_bfloat16* B;
  const __nv_bfloat16* w_g;
  float b_g, alpha;
  int gh;                   // vector-gate hidden width (0: the scalar gate)
  const float *gw1, *gc1, *gw2, *gc2;
  float* ws_P;              // [NP][r + 4]: (A x)[j] for j < r, w_g . x at j = r (16-byte rows)
  uint4* ws_T;              // [NP][r / 4]: T hi/lo, pairs (2q, 2q + 1) of token m at m r / 4 + q
  unsigned* ws_sync;        // [0] producer row tiles published, [1] tile-CTA ticket, [2] T published
  uint32_t off_bf, off_x16, off_xr, off_B;   // dynamic shared memory layout
  uint64_t t_wait_ns;       // limit of the wait for the published T
};

__device__ __forceinline__ void give_up(int* abort_flag) {
  record_status(&g_dtc_status, DEV_ERR_TIMEOUT);
  atomicExch(abort_flag, 1);
}

// ------------------------------------------------------------- producers --
// The producer CTA that publishes the last row tile of P forms T for every
// token, with all of its threads and long before the tile CTAs need it:
//   scalar gate  T[m] = alpha g_m t_m,        g_m = sigmoid(P[m][r] + b_g)
//   vector gate  T[m] = alpha gamma(t_m) t_m  (the bottleneck MLP on t_m)
// with t_m = P[m][0 .. r) and T = 0 for tokens m >= M, split into bf16 hi +
// lo (T = hi + lo to ~2^-16 relative) in the pair order of the epilogue's
// B operand, and published with ws_sync[2].
template <int NP>
__device__ __noinline__ void tc_form_T(const TcParams& p, uint8_t* smem) {
  const int r = p.r, ps = r + 4, r4 = r / 4;
  float* ts = reinterpret_cast<float*>(smem);               // [NP][r]
  float* gl = ts + NP * r;                                   // [NP] gate logits (scalar gate)
  float* gsm = gl + NP;                                      // gate weights (vector gate), 16-byte aligned
  float* hid = gsm + (p.gh > 0 ? gate_smem_floats(r, p.gh) : 0);   // [NP][h | 1]
  if (p.gh > 0) stage_gate_weights_async(p.gw1, p.gw2, p.gc1, p.gc2, r, p.gh, gsm, threadIdx.x, kThreads);
  for (int e = threadIdx.x; e < NP * r4; e += kThreads)
    reinterpret_cast<float4*>(ts)[e] = __ldcg(reinterpret_cast<const float4*>(p.ws_P + (size_t)(e / r4) * ps) + e % r4);
  for (int m = threadIdx.x; m < NP; m += kThreads) gl[m] = __ldcg(p.ws_P + (size_t)m * ps + r);
  if (p.gh > 0) cp_async_wait<0>();
  __syncthreads();
  if (p.gh > 0) {
    const GateSmem g(gsm, r, p.gh);
    vector_gate_hidden_rows(ts, NP, g, hid, threadIdx.x, kThreads);
    __syncthreads();
    vector_gate_apply_rows(ts, NP, g, hid, threadIdx.x, kThreads);     // t *= gamma(t)
    __syncthreads();
  }
  for (int e = threadIdx.x; e < NP * r4; e += kThreads) {
    const int m = e / r4;
    const float gm = m >= p.M ? 0.0f : p.gh > 0 ? p.alpha : p.alpha / (1.0f + expf(-(gl[m] + p.b_g)));
    const float4 tv = reinterpret_cast<const float4*>(ts)[e];
    const float t0 = gm * tv.x, t1 = gm * tv.y, t2 = gm * tv.z, t3 = gm * tv.w;
    const float h0 = __bfloat162float(__float2bfloat16_rn(t0)), h1 = __bfloat162float(__float2bfloat16_rn(t1));
    const float h2 = __bfloat162float(__float2bfloat16_rn(t2)), h3 = __bfloat162float(__float2bfloat16_rn(t3));
    __stcg(p.ws_T + e, make_uint4(pack_bf16x2(h0, h1), pack_bf16x2(t0 - h0, t1 - h1),
                                  pack_bf16x2(h2, h3), pack_bf16x2(t2 - h2, t3 - h3)));
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicExch(&p.ws_sync[2], 1u);
  }
}

// Producer cluster rt (a 16-row tile of [A; w_g]): CTA `rank` of it covers K
// slice `rank` of S (128-k chunks).  Lane (g, c) of a warp loads
// 8 consecutive k of a projection row and of a token; both operands use the
// same k permutation, so the mma.sync sums are the plain dot products.
template <int NP>
__device__ void tc_producer(const TcParams& p, uint8_t* smem, int rt, int rank) {
  constexpr int MT = NP / 8;
  constexpr int NW = kThreads / 32;
  constexpr int U = MT <= 2 ? 2 : 1;                       // 32-k pieces per pass
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int nch = p.K / 128;
  const int c0 = (int)((long long)rank * nch / p.S), c1 = (int)((long long)(rank + 1) * nch / p.S);
  const int npieces = (c1 - c0) * 4;
  float* red = reinterpret_cast<float*>(smem);             // [NW][MT][4][32]
  float* part = red + NW * MT * 128;                        // [16][NP]

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
  // the rows of A and w_g are weights: the first pass loads them before
  // waiting for the kernel ahead (overlapped launches), then the tokens
  bool waited = false;
  for (int pc0 = warp; pc0 < npieces; pc0 += U * NW) {
    uint4 va[U], vb[U], xv[U][MT];
#pragma unroll
    for (int h = 0; h < U; ++h) {
      const int pcs = pc0 + h * NW;
      const bool ok = pcs < npieces;
      const int kb = c0 * 128 + pcs * 32 + 8 * c;
      va[h] = (ok && wlo) ? ldg16(wlo + kb) : make_uint4(0, 0, 0, 0);
      vb[h] = (ok && whi) ? ldg16(whi + kb) : make_uint4(0, 0, 0, 0);
    }
    if (!waited) {
      pdl_wait();
      waited = true;
    }
#pragma unroll
    for (int h = 0; h < U; ++h) {
      const int pcs = pc0 + h * NW;
      const bool ok = pcs < npieces;
      const int kb = c0 * 128 + pcs * 32 + 8 * c;
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        const int tok = t * 8 + g;
        xv[h][t] = (ok && tok < p.M) ? ldg16(p.x + (size_t)tok * p.K + kb) : make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int h = 0; h < U; ++h)
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        mma_bf16_16816(acc[t], va[h].x, vb[h].x, va[h].y, vb[h].y, xv[h][t].x, xv[h][t].y);
        mma_bf16_16816(acc[t], va[h].z, vb[h].z, va[h].w, vb[h].w, xv[h][t].z, xv[h][t].w);
      }
  }
  if (!waited) pdl_wait();                                 // before the workspace
  // fixed-order sum over the warps: this CTA's partial [16 rows][NP tokens]
#pragma unroll
  for (int t = 0; t < MT; ++t)
#pragma unroll
    for (int i = 0; i < 4; ++i) red[((warp * MT + t) * 4 + i) * 32 + lane] = acc[t][i];
  __syncthreads();
  for (int e = threadIdx.x; e < MT * 128; e += kThreads) {
    const int t = e / 128, i = (e / 32) & 3, ln = e & 31;
    float v = 0.0f;
    for (int w = 0; w < NW; ++w) v += red[((w * MT + t) * 4 + i) * 32 + ln];
    // C fragment element i of lane ln: row (ln/4) + 8 (i/2), token t*8 + 2 (ln%4) + (i%2)
    part[((ln >> 2) + 8 * (i >> 1)) * NP + t * 8 + 2 * (ln & 3) + (i & 1)] = v;
  }
  __syncthreads();
  cluster_sync();                                          // every CTA's partial is in its shared memory

  if (rank == 0) {
    // the S partials in rank order (every load in flight, then the sum), then
    // row tile rt of P is published
    SPEAR_CHECK(&g_dtc_status, rt < p.RT && p.S <= kMaxS);
    for (int e = threadIdx.x; e < 16 * NP; e += kThreads) {
      const uint32_t la = smem_u32(part + e);
      float pv[kMaxS];
#pragma unroll
      for (int q = 0; q < kMaxS; ++q)
        if (q < p.S) pv[q] = dsmem_ld_f32(dsmem_addr(la, (uint32_t)q));
      float v = 0.0f;
#pragma unroll
      for (int q = 0; q < kMaxS; ++q)
        if (q < p.S) v += pv[q];
      const int row = e / NP, tok = e % NP, i = rt * 16 + row;
      if (i <= p.r) p.ws_P[(size_t)tok * (p.r + 4) + i] = v;
    }
    __syncthreads();
    __shared__ int s_last;
    if (threadIdx.x == 0) {
      __threadfence();
      s_last = atomicAdd(&p.ws_sync[0], 1u) == (unsigned)(p.RT - 1);
      __threadfence();                                     // every row tile of P is visible from here
    }
    __syncthreads();
    if (s_last) tc_form_T<NP>(p, smem);                    // this CTA's shared memory is no longer read
  }
  cluster_sync();                                          // peers keep their shared memory until read
}

// ---------------------------------------------------------- tile CTAs --
// The K units (256 k) of tile CTA `rank` of a cluster of S: rank, rank + S,
// rank + 2 S, ... (the cluster walks each row's bytes together); the last
// unit of K may hold only 128 k.  When U = b S + q units leave q CTAs one unit
// longer than the rest and 2 q <= S (and K has no such tail), each of those q
// units is split: its CTA keeps the first 128 k and CTA q + j takes the second
// 128 k as one more unit, so no CTA carries more than b + 1/2 units.
struct TcUnits {
  int n;          // units of this CTA
  bool half;      // its last unit holds 128 k
  int k0_extra;   // k of a second-half unit taken from another CTA (its last), or -1
  int kbase, kstride;
  __device__ TcUnits(int units, int K, int rank, int S) : kbase(rank * kUnitK), kstride(S * kUnitK) {
    const int b = units / S, q = units % S;
    const bool ktail = (K % kUnitK) != 0;
    const bool split = !ktail && q > 0 && 2 * q <= S;
    const bool takes = split && rank >= q && rank < 2 * q;
    n = (units - rank + S - 1) / S + (takes ? 1 : 0);
    half = (ktail && (units - 1) % S == rank) || (split && rank < 2 * q);
    k0_extra = takes ? (b * S + rank - q) * kUnitK + kUnitK / 2 : -1;
  }
  __device__ int k0(int i) const { return (k0_extra >= 0 && i == n - 1) ? k0_extra : kbase + i * kstride; }
  __device__ int len(int i) const { return (half && i == n - 1) ? kUnitK / 2 : kUnitK; }
};

// Rows n and n + 32 of the tile's partial for token t, computed in fp32 over
// the CTA's K units from the int4 codes and the bf16 token: the path for a
// token with a value beyond the fp16 range (the tensor core would see inf).
// Each weight is formed as the converters form it (u - z exact, times the
// group scale with one fp16 rounding; per-channel: u - z, the scale applied
// to the sum), so only the summation order differs from the tensor-core path.
template <bool PERCH>
__device__ __forceinline__ void tc_exact_rows(const TcParams& p, float* red, const float* s_scale, int n, int t,
                                           const TcUnits& us) {
  const int zrow = (p.ng + 1) / 2;
  const int row0 = n % kTileRows;
  const __nv_bfloat16* xt = p.x + (size_t)t * p.K;
  float acc[2] = {0.0f, 0.0f};
  bool nonfinite = false;
  for (int i = 0; i < us.n; ++i) {
    const int k0 = us.k0(i), k1 = min(p.K, k0 + us.len(i));
    for (int k = k0; k < k1; k += 32) {
      float xf[32];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(xt + k) + j);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          xf[8 * j + 2 * e] = __uint_as_float(w[e] << 16);
          xf[8 * j + 2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
        }
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) nonfinite |= !(fabsf(xf[j]) <= 3.402823466e38f);
      const int g = PERCH ? 0 : k / 128;
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int nn = n + 32 * rr;
        if (nn >= p.N) continue;
        const uint32_t zb = p.sym ? 0x88u : (uint32_t)__ldg(p.zeros + (size_t)nn * zrow + g / 2);
        const int z = (int)((g & 1) ? (zb >> 4) : (zb & 15u));
        const __half sc = PERCH ? __float2half(1.0f) : __ldg(p.scales + (size_t)nn * p.ng + g);
        const uint4 cv = __ldg(reinterpret_cast<const uint4*>(p.qweight + (size_t)nn * (p.K / 2) + k / 2));
        const uint32_t cw[4] = {cv.x, cv.y, cv.z, cv.w};
        float a = acc[rr];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int u = (int)((cw[j >> 3] >> (4 * (j & 7))) & 15u);
          const float wv = PERCH ? (float)(u - z) : __half2float(__hmul(__int2half_rn(u - z), sc));
          a = fmaf(wv, xf[j], a);
        }
        acc[rr] = a;
      }
    }
  }
  if (nonfinite) record_status(&g_dtc_status, DEV_ERR_INVALID);   // inf or NaN among the token's values
#pragma unroll
  for (int rr = 0; rr < 2; ++rr)
    red[t * kRedStride + row0 + 32 * rr] = (n + 32 * rr < p.N) ? s_scale[row0 + 32 * rr] * acc[rr] : 0.0f;
}

// One CTA = 256 weight rows x its K units.  The tensor core sees the tokens
// as the 64-row A operand (M = 64: accumulator row m lives in TMEM lane
// (m mod 16) + 32 (m / 16)) and the weights as the 256-column B operand, so
// one instruction covers 256 rows x 16 k of int4.  Within each 8-k chunk both
// operands hold k in the order 0,4,1,5,2,6,3,7: the order in which the
// converters take nibble pairs out of a 32-bit word; every 16-k MMA still
// sums the same products.
template <int NP, bool PERCH, bool COMP>
__device__ void tc_tile(const CUtensorMap* tm_w, const CUtensorMap* tm_x, const TcParams& p, uint8_t* smem,
                        int tile, int rank) {
  __shared__ __align__(8) uint64_t raw_full[kRawStages], raw_empty[kRawStages];
  __shared__ __align__(8) uint64_t xr_full[kXrStages], xr_empty[kXrStages];
  __shared__ __align__(8) uint64_t x16_full[kX16Stages], x16_empty[kX16Stages];
  __shared__ __align__(8) uint64_t bf_full[kMaxBfStages], bf_empty[kMaxBfStages];
  __shared__ __align__(8) uint64_t acc_full;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_pok;
  __shared__ unsigned s_big[2];   // tokens whose fp16 copy overflowed on this CTA's K range (bit t)
  unsigned ticket = 0;            // thread 0: this CTA's place among the tile CTAs past the P wait
  __shared__ float s_scale[kTileRows];                     // per-channel scales of the tile rows

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.S, BF = p.bf_stages;
  const int n0 = tile * kTileRows;
  // K units of this CTA (TcUnits)
  const TcUnits us(p.units, p.K, rank, S);
  const int nunits = us.n;
  const int nsteps = 4 * nunits - (us.half ? 2 : 0);       // 64-k steps (even)
  const int ngroups = nsteps / 2;                          // 128-k groups
  // rows finished here: whole 16-row tiles, so every owner range starts on a
  // 16-byte boundary of the partial and of y
  const int e_r0 = 16 * (rank * (kTileRows / 16) / S), e_r1 = 16 * ((rank + 1) * (kTileRows / 16) / S);
  const int nr = e_r1 - e_r0;

  uint8_t* raw_ring = smem;                                // [2][256 rows][128 B] int4
  uint8_t* bf_ring = smem + p.off_bf;                      // [BF][256 rows][128 B] fp16 weights
  uint8_t* x16_ring = smem + p.off_x16;                    // [3][64 tokens][128 B] fp16 tokens
  uint8_t* xr_ring = smem + p.off_xr;                      // [2][NP tokens][128 B] bf16 tokens (TMA)
  uint8_t* B_s = smem + p.off_B;                           // [nr][2r + 16 bytes]
  // after the main loop: the partial [64 tokens][260] over the raw ring and
  // the start of the weight ring
  float* red = reinterpret_cast<float*>(smem);
  // T = alpha g t split into bf16 hi + lo (T = hi + lo to ~2^-16 relative),
  // the B operand of the epilogue's B T on warp-level MMAs: in the bf16 token
  // ring once the last token tile is converted (NP r 4 <= 2 NP 128 bytes);
  // element (m, jj) holds the hi and the lo bf16 pair of T[m][2jj .. 2jj+1]
  uint2* thl_s = reinterpret_cast<uint2*>(xr_ring);                 // [NP][r/2]
  const int b_stride = 2 * p.r + 16;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kRawStages; ++i) {
      mbar_init(smem_u32(&raw_full[i]), 1);
      mbar_init(smem_u32(&raw_empty[i]), kConvWarps);
    }
    for (int i = 0; i < kXrStages; ++i) {
      mbar_init(smem_u32(&xr_full[i]), 1);
      mbar_init(smem_u32(&xr_empty[i]), kXWarps);
    }
    for (int i = 0; i < kX16Stages; ++i) {
      mbar_init(smem_u32(&x16_full[i]), kXWarps);
      mbar_init(smem_u32(&x16_empty[i]), 1);
    }
    for (int i = 0; i < kMaxBfStages; ++i) {
      mbar_init(smem_u32(&bf_full[i]), kConvWarps);
      mbar_init(smem_u32(&bf_empty[i]), 1);
    }
    mbar_init(smem_u32(&acc_full), 1 + kXWarps);          // the last commit and the token warps' flags
    s_abort = 0;
    s_pok = 0;
    s_big[0] = s_big[1] = 0u;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&s_tmem), kTileRows);
    tmem_relinquish();
  }
  if (warp < kXWarps) {
    // token rows NP..63 of every fp16 token slot stay zero
    if constexpr (NP < 64) {
      constexpr int kPad = (64 - NP) * 8;                  // 16-byte chunks per slot
      for (int i = threadIdx.x; i < kX16Stages * kPad; i += kXWarps * 32)
        *reinterpret_cast<uint4*>(x16_ring + (i / kPad) * kX16Bytes + NP * 128 + (i % kPad) * 16) =
            make_uint4(0, 0, 0, 0);
    }
    for (int r = threadIdx.x; r < kTileRows; r += kXWarps * 32)
      s_scale[r] = (PERCH && n0 + r < p.N) ? __half2float(__ldg(p.scales + (size_t)(n0 + r) * p.ng)) : 1.0f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------- TMA
    // The whole warp runs the loop (lane 0 tests the slots and issues, the
    // decisions are broadcast), like the MMA warp below.
    if (lane == 0) {
      prefetch_tmap(tm_w);
      prefetch_tmap(tm_x);
      SPEAR_CHECK(&g_dtc_status, n0 < p.N && (nunits == 0 || us.k0(nunits - 1) < p.K));
    }
    // the first weight units need no slot wait and read only the layer's
    // weights: issue them before waiting for the kernel ahead (overlapped launches)
    int ri = nunits < kRawStages ? nunits : kRawStages, xi = 0;
    if (lane == 0) {
      for (int i = 0; i < ri; ++i) {
        const uint32_t full = smem_u32(&raw_full[i]);
        mbar_arrive_expect_tx(full, kRawBytes);
        tma_load_2d(smem_u32(raw_ring + i * kRawBytes), tm_w, us.k0(i) >> 1, n0, full);
      }
    }
    __syncwarp();
    pdl_wait();
    bool ok = true;
    uint64_t t0 = globaltimer_ns();
    uint32_t idle = 0;
    while (ok && (ri < nunits || xi < nsteps)) {
      uint32_t prog = 0;
      if (lane == 0) {
        if (ri < nunits) {
          const int slot = ri % kRawStages;
          if (mbar_test_wait(smem_u32(&raw_empty[slot]), ((ri / kRawStages) & 1) ^ 1)) {
            const uint32_t full = smem_u32(&raw_full[slot]);
            mbar_arrive_expect_tx(full, kRawBytes);
            tma_load_2d(smem_u32(raw_ring + slot * kRawBytes), tm_w, us.k0(ri) >> 1, n0, full);
            prog |= 1u;
          }
        }
        if (xi < nsteps) {
          const int slot = xi % kXrStages;
          if (mbar_test_wait(smem_u32(&xr_empty[slot]), ((xi / kXrStages) & 1) ^ 1)) {
            const uint32_t full = smem_u32(&xr_full[slot]);
            mbar_arrive_expect_tx(full, NP * 128);
            tma_load_2d(smem_u32(xr_ring + slot * NP * 128), tm_x, us.k0(xi >> 2) + (xi & 3) * kStepK,
                        0, full);
            prog |= 2u;
          }
        }
      }
      prog = __shfl_sync(0xffffffffu, prog, 0);
      ri += (int)(prog & 1u);
      xi += (int)(prog >> 1);
      if (prog) {
        idle = 0;
      } else {
        __nanosleep(64);                                   // leave the issue slots to the converters
        if ((++idle & 63) == 0) {
          if (idle == 64) t0 = globaltimer_ns();
          else if (globaltimer_ns() - t0 > kPipeWaitNs || s_abort) ok = false;
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        }
      }
    }
    if (!ok && lane == 0) {
      give_up(&s_abort);
      // never leave with copies in flight: wait (bounded) for every issued fill
      for (int i = std::max(0, ri - kRawStages); i < ri; ++i)
        mbar_wait(smem_u32(&raw_full[i % kRawStages]), (i / kRawStages) & 1, kPipeWaitNs);
      for (int i = std::max(0, xi - kXrStages); i < xi; ++i)
        mbar_wait(smem_u32(&xr_full[i % kXrStages]), (i / kXrStages) & 1, kPipeWaitNs);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------- MMA
    // The whole warp runs the loop (every lane waits, one elected lane
    // issues): a loop on one lane while the other 31 wait at a barrier issues
    // at about a third of the rate.
    const uint32_t idesc = idesc_f16_f32(64, kTileRows);
    bool ok = true;
    for (int s = 0; s < nsteps; ++s) {
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bf_full[s % BF]), (s / BF) & 1, kPipeWaitNs) &&
                                       mbar_wait(smem_u32(&x16_full[s % kX16Stages]), (s / kX16Stages) & 1,
                                                 kPipeWaitNs) && !s_abort);
      if (!ok) {
        if (lane == 0) give_up(&s_abort);
        break;
      }
      tc_fence_after();
      const uint32_t a0 = smem_u32(x16_ring + (s % kX16Stages) * kX16Bytes);
      const uint32_t b0 = smem_u32(bf_ring + (s % BF) * kBfBytes);
#pragma unroll
      for (int kk = 0; kk < kStepK / 16; ++kk)
        mma_bf16_ss_warp(tmem, smem_desc(a0 + 32 * kk, 1024, LAYOUT_SW128),
                         smem_desc(b0 + 32 * kk, 1024, LAYOUT_SW128), idesc, (s > 0 || kk > 0) ? 1u : 0u);
      mma_commit_warp(smem_u32(&bf_empty[s % BF]));
      mma_commit_warp(smem_u32(&x16_empty[s % kX16Stages]));
    }
    if (ok) mma_commit_warp(smem_u32(&acc_full));
  } else if (warp >= kConvWarp0) {
    // -------------------------------------- weight converters (16 warps)
    const int cw = warp - kConvWarp0;
    const int half = cw >> 3;
    const int row = 32 * (cw & 7) + lane;                  // 0..255
    const int n = n0 + row;
    const bool row_ok = n < p.N;
    const int zrow = (p.ng + 1) / 2;
    auto gidx = [&](int gl) { return PERCH ? 0 : (us.k0(gl >> 1) >> 7) + (gl & 1); };
    // The prefetched registers hold the loaded zero-point byte and scale bits
    // as they are; the nibble is picked and the scale doubled where they are
    // used, so no instruction waits for the load before then.
    auto load_z = [&](int gl) -> uint32_t {
      if (p.sym || !row_ok || gl >= ngroups) return 0x88u;
      return __ldg(p.zeros + (size_t)n * zrow + gidx(gl) / 2);
    };
    auto load_s = [&](int gl) -> uint32_t {
      if (PERCH || !row_ok || gl >= ngroups) return 0u;
      return __half_as_ushort(__ldg(p.scales + (size_t)n * p.ng + gidx(gl)));
    };
    bool ok = true;
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      ok = __all_sync(0xffffffffu, ok && mbar_wait(smem_u32(bar), parity, kPipeWaitNs) && !s_abort);
    };
    // one 64-k step: this thread's 32 k of its row, as (u - z) * s in fp16
    auto convert = [&](int s, uint32_t zb, uint32_t sb) {
      const int u = s >> 2, j = s & 3, slot = u % kRawStages;
      if (j == 0) wait_all(&raw_full[slot], (u / kRawStages) & 1);
      wait_all(&bf_empty[s % BF], ((s / BF) & 1) ^ 1);
      if (ok) {
        const uint32_t z = (gidx(s >> 1) & 1) ? (zb >> 4) : (zb & 15u);
        const uint32_t s2 = sb * 0x00010001u;                      // fp16x2 of the group scale
        const uint4 rv = *reinterpret_cast<const uint4*>(raw_ring + slot * kRawBytes + row * 128 +
                                                          (((2 * j + half) ^ (row & 7)) << 4));
        uint8_t* brow = bf_ring + (s % BF) * kBfBytes + row * 128;
        const uint32_t z_lo = f16x2_bias(z);                       // 1024 + z
        const uint32_t z_hi = (0x5400u | (z << 4)) * 0x00010001u;  // 64 + z
        const uint32_t words[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint32_t a = words[w], b = words[w] >> 8;
          // (k0,k4) and (k2,k6) as 1024 + u; (k1,k5) and (k3,k7) as 64 + u (the
          // nibble left in place, one fp16 mantissa unit = 1/16 at 64)
          uint32_t v0 = (a & 0x000F000Fu) | 0x64006400u, v1 = (a & 0x00F000F0u) | 0x54005400u;
          uint32_t v2 = (b & 0x000F000Fu) | 0x64006400u, v3 = (b & 0x00F000F0u) | 0x54005400u;
          v0 = f16x2_sub(v0, z_lo); v2 = f16x2_sub(v2, z_lo);     // exact u - z
          v1 = f16x2_sub(v1, z_hi); v3 = f16x2_sub(v3, z_hi);
          if (!PERCH) { v0 = f16x2_mul(v0, s2); v1 = f16x2_mul(v1, s2); v2 = f16x2_mul(v2, s2); v3 = f16x2_mul(v3, s2); }
          *reinterpret_cast<uint4*>(brow + (((4 * half + w) ^ (row & 7)) << 4)) = make_uint4(v0, v1, v2, v3);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&bf_full[s % BF]));
        if (j == 3 || s == nsteps - 1) mbar_arrive(smem_u32(&raw_empty[slot]));
      }
    };
    // the factor-B rows of the rows finished here, for the epilogue: in
    // flight during the conversions
    if (COMP) {
      const int per = p.r / 8;                             // 16-byte pieces per row
      for (int e = threadIdx.x - kConvWarp0 * 32; e < nr * per; e += kConvWarps * 32) {
        const int rr = e / per, cc = e % per, nn = n0 + e_r0 + rr;
        if (nn < p.N) cp_async16(B_s + rr * b_stride + cc * 16, p.B + (size_t)nn * p.r + cc * 8);
      }
      cp_async_commit();
    }
    // zero points and scales travel 4 groups ahead of their use in named
    // registers (slot = group mod 4, never indexed at run time)
    uint32_t z0 = load_z(0), z1 = load_z(1), z2 = load_z(2), z3 = load_z(3);
    uint32_t c0 = load_s(0), c1 = load_s(1), c2 = load_s(2), c3 = load_s(3);
    auto group = [&](int gl, uint32_t& zs, uint32_t& cs) {
      convert(2 * gl, zs, cs);
      convert(2 * gl + 1, zs, cs);
      zs = load_z(gl + 4);
      cs = load_s(gl + 4);
    };
    for (int gl0 = 0; gl0 < ngroups; gl0 += 4) {
      if (gl0 + 0 < ngroups) group(gl0 + 0, z0, c0);
      if (gl0 + 1 < ngroups) group(gl0 + 1, z1, c1);
      if (gl0 + 2 < ngroups) group(gl0 + 2, z2, c2);
      if (gl0 + 3 < ngroups) group(gl0 + 3, z3, c3);
    }
    if (COMP) cp_async_wait<0>();

    // accumulator [64 tokens][256 rows] -> this CTA's partial, token-major (row
    // stride 257).  Each converter warp drains 64 columns of the TMEM lane
    // quarter it may access (warp mod 4); tokens 16 q .. 16 q + 15 sit in its
    // lanes 0-15.
    ok = __all_sync(0xffffffffu, ok && mbar_wait(smem_u32(&acc_full), 0, kPipeWaitNs) && !s_abort);
    if (ok) {
      tc_fence_after();
      const int q = warp & 3, cb = 64 * ((warp - kConvWarp0) >> 2);
      const int t = 16 * q + lane;
      const bool t_ok = lane < 16 && t < NP;
#pragma unroll 1
      for (int c0 = cb; c0 < cb + 64; c0 += 32) {
        uint32_t v[32];
        tmem_ld_32cols(tmem + ((uint32_t)(32 * q) << 16) + c0, v);
        tmem_ld_wait();
        if (t_ok) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(red + t * kRedStride + c0 + i) =
                make_float4(s_scale[c0 + i] * __uint_as_float(v[i]), s_scale[c0 + i + 1] * __uint_as_float(v[i + 1]),
                            s_scale[c0 + i + 2] * __uint_as_float(v[i + 2]),
                            s_scale[c0 + i + 3] * __uint_as_float(v[i + 3]));
        }
      }
      // tokens of this warp whose fp16 copy overflowed: their rows of the
      // partial are recomputed here in fp32 (the flags were set before the
      // token warps arrived on acc_full)
      const uint32_t big16 = (s_big[q >> 1] >> (16 * (q & 1))) & 0xFFFFu;
      if (big16 != 0u) {
        __syncwarp();
        for (uint32_t b = big16; b != 0u; b &= b - 1u)
          tc_exact_rows<PERCH>(p, red, s_scale, n0 + cb + lane, 16 * q + (__ffs(b) - 1), us);
      }
    } else {
      give_up(&s_abort);
    }
  } else {
    // --------------------------- token converters + epilogue (warps 0-3)
    const int tid = threadIdx.x;                           // 0..127
    pdl_wait();                                            // they read the workspace
    bool ok = true;
    uint32_t bigm = 0;                                     // bit i: chunk tid + 128 i held |x| >= 65504
    for (int s = 0; s < nsteps; ++s) {
      const int rs = s % kXrStages, xs = s % kX16Stages;
      ok = ok && mbar_wait(smem_u32(&xr_full[rs]), (s / kXrStages) & 1, kPipeWaitNs) &&
           mbar_wait(smem_u32(&x16_empty[xs]), ((s / kX16Stages) & 1) ^ 1, kPipeWaitNs);
      ok = __all_sync(0xffffffffu, ok && !s_abort);
      if (ok) {
        const uint8_t* src = xr_ring + rs * NP * 128;
        uint8_t* dst = x16_ring + xs * kX16Bytes;
#pragma unroll
        for (int i = 0; i < NP * 8 / (kXWarps * 32); ++i) {
          // 16-byte chunk c: token c / 8, k 8 (c % 8) .. +7; same swizzled place in both tiles
          const int c = tid + i * (kXWarps * 32), t = c >> 3, off = t * 128 + (((c & 7) ^ (t & 7)) << 4);
          const uint4 v = *reinterpret_cast<const uint4*>(src + off);
          const float x0 = bf16x2_lo(v.x), x1 = bf16x2_hi(v.x), x2 = bf16x2_lo(v.y), x3 = bf16x2_hi(v.y);
          const float x4 = bf16x2_lo(v.z), x5 = bf16x2_hi(v.z), x6 = bf16x2_lo(v.w), x7 = bf16x2_hi(v.w);
          const float m = fmaxf(fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3))),
                                fmaxf(fmaxf(fabsf(x4), fabsf(x5)), fmaxf(fabsf(x6), fabsf(x7))));
          bigm |= (m < 65504.0f ? 0u : 1u) << i;
          auto h2 = [](float lo, float hi) {
            const __half2 h = __floats2half2_rn(lo, hi);
            return *reinterpret_cast<const uint32_t*>(&h);
          };
          *reinterpret_cast<uint4*>(dst + off) = make_uint4(h2(x0, x4), h2(x1, x5), h2(x2, x6), h2(x3, x7));
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&x16_full[xs]));
        mbar_arrive(smem_u32(&xr_empty[rs]));
      }
    }
    // tokens whose fp16 copy overflowed somewhere in this CTA's K range
    for (uint32_t b = bigm; b != 0u; b &= b - 1u) {
      const int t = (tid + (kXWarps * 32) * (__ffs(b) - 1)) >> 3;
      atomicOr(&s_big[t >> 5], 1u << (t & 31));
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&acc_full));      // the overflow flags are in place

    if (COMP) {
      // T hi/lo as the last producer published it, copied into the spent
      // token ring (one round trip: every load of a thread in flight together)
      if (tid == 0) {
        const uint64_t tw = globaltimer_ns();
        int pok = 0;
        for (unsigned i = 0;; ++i) {
          if (ld_acquire_gpu(&p.ws_sync[2]) != 0u) { pok = 1; break; }
          if ((i & 63) == 63 && globaltimer_ns() - tw > p.t_wait_ns) break;
          __nanosleep(64);
        }
        if (!pok) record_status(&g_dtc_status, DEV_ERR_TIMEOUT);
        s_pok = pok;
        // taken here, read at the end of the kernel: the round trip overlaps
        // the rest of the work
        ticket = atomicAdd(&p.ws_sync[1], 1u);
      }
      named_sync(1, kXWarps * 32);
      const bool pok = s_pok != 0;
      const int n4 = NP * p.r / 4;                         // 16-byte pieces of T hi/lo
      constexpr int kPerQ = 4;
      for (int e0 = 0; e0 < n4; e0 += kPerQ * kXWarps * 32) {
        uint4 v[kPerQ];
#pragma unroll
        for (int i = 0; i < kPerQ; ++i) v[i] = __ldcg(p.ws_T + min(e0 + tid + i * kXWarps * 32, n4 - 1));
#pragma unroll
        for (int i = 0; i < kPerQ; ++i) {
          const int e = e0 + tid + i * kXWarps * 32;
          if (e < n4) reinterpret_cast<uint4*>(thl_s)[e] = pok ? v[i] : make_uint4(0u, 0u, 0u, 0u);
        }
      }
    }
  }

  // ---------------------------------------------- epilogue (whole cluster)
  if (COMP && warp < kTmaWarp) {
    // B T for the rows finished here, added into this CTA's own partial
    // before the cluster reads it: one (16-row, 8-token) tile per warp at a
    // time on mma.sync (B rows as A, T hi/lo as B).  Warps 0-19 only: the
    // TMA and MMA warps never reach this barrier.
    named_sync(2, kTmaWarp * 32);                          // drained partial, T and B rows in place
    if (!s_abort) {
      const int g = lane >> 2, c = lane & 3;
      const int rtiles = nr / 16, ttiles = (p.M + 7) / 8;
      for (int item = warp; item < rtiles * ttiles; item += kTmaWarp) {
        const int rt = item % rtiles, tt = item / rtiles;
        float bt[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        const uint8_t* blo = B_s + (rt * 16 + g) * b_stride;
        const uint8_t* bhi = blo + 8 * b_stride;
        const int tok = tt * 8 + g;
        const uint2* thl = thl_s + tok * (p.r / 2);
        for (int j0 = 0; j0 < p.r; j0 += 16) {
          const uint32_t a0 = *reinterpret_cast<const uint32_t*>(blo + (j0 + 2 * c) * 2);
          const uint32_t a1 = *reinterpret_cast<const uint32_t*>(bhi + (j0 + 2 * c) * 2);
          const uint32_t a2 = *reinterpret_cast<const uint32_t*>(blo + (j0 + 2 * c + 8) * 2);
          const uint32_t a3 = *reinterpret_cast<const uint32_t*>(bhi + (j0 + 2 * c + 8) * 2);
          const uint2 t0 = thl[j0 / 2 + c], t1 = thl[j0 / 2 + c + 4];
          mma_bf16_16816(bt, a0, a1, a2, a3, t0.x, t1.x);
          mma_bf16_16816(bt, a0, a1, a2, a3, t0.y, t1.y);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int rl = rt * 16 + g + 8 * (i >> 1), t = tt * 8 + 2 * c + (i & 1);
          if (t < p.M) red[t * kRedStride + e_r0 + rl] += bt[i];
        }
      }
    }
  }
  pdl_wait();                                              // y may be read by the kernel ahead
  cluster_sync();                                          // every partial is in place
  if (!s_abort) {
    // y for the rows finished here: four consecutive rows of one token per
    // thread, the S partials read 16 bytes at a time (all in flight), summed
    // in rank order
    const uint32_t red_base = smem_u32(red);
    const int nq = nr / 4;
    const bool vec = (p.N & 3) == 0;
    for (int idx = threadIdx.x; idx < p.M * nq; idx += kThreads) {
      const int t = idx / nq, row = e_r0 + 4 * (idx % nq), nn = n0 + row;
      const uint32_t la = red_base + (uint32_t)(t * kRedStride + row) * 4u;
      float4 pv[kMaxS];
#pragma unroll
      for (int qq = 0; qq < kMaxS; ++qq)
        if (qq < S) pv[qq] = dsmem_ld_f32x4(dsmem_addr(la, (uint32_t)qq));
      float4 v = pv[0];
#pragma unroll
      for (int qq = 1; qq < kMaxS; ++qq)
        if (qq < S) { v.x += pv[qq].x; v.y += pv[qq].y; v.z += pv[qq].z; v.w += pv[qq].w; }
      if (nn >= p.N) continue;
      const size_t o = (size_t)t * p.N + nn;
      SPEAR_CHECK(&g_dtc_status, t < p.M && nn < p.N && (!vec || nn + 3 < p.N));
      if (vec) {                                           // nn + 3 < N as N and nn are multiples of 4
        if (p.out_f32) {
          *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.y) + o) = v;
        } else {
          const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
          uint2 pk;
          pk.x = *reinterpret_cast<const uint32_t*>(&lo);
          pk.y = *reinterpret_cast<const uint32_t*>(&hi);
          *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.y) + o) = pk;
        }
      } else {
        const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (nn + j >= p.N) break;
          if (p.out_f32) reinterpret_cast<float*>(p.y)[o + j] = vv[j];
          else reinterpret_cast<__nv_bfloat16*>(p.y)[o + j] = __float2bfloat16_rn(vv[j]);
        }
      }
    }
  }
  if (COMP && threadIdx.x == 0 && ticket == (unsigned)(p.n_consumers - 1)) {   // every tile CTA has seen P
    p.ws_sync[1] = 0;
    p.ws_sync[2] = 0;
    atomicExch(&p.ws_sync[0], 0u);
  }
  tc_fence_before();
  cluster_sync();                                          // peers are done reading this CTA
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTileRows);
  }
}

template <int NP, bool PERCH, bool COMP>
__global__ void __launch_bounds__(kThreads, 1)
decode_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                 const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align_up(smem_raw, 1024);
  pdl_launch_dependents();                                 // every CTA is resident: let the next kernel queue
  const int rank = (int)cluster_ctarank();
  const int cid = (int)blockIdx.x / p.S;
  const int npc = p.RT;
  if (cid < npc) {
    // producer clusters; with the compensator off they idle (the tile split
    // stays the one of the compensated layer, so a zero gate reproduces the
    // plain layer bit for bit)
    if (COMP) tc_producer<NP>(p, smem, cid, rank);
    return;
  }
  tc_tile<NP, PERCH, COMP>(&tm_w, &tm_x, p, smem, cid - npc, rank);
}

using TcKernel = void (*)(CUtensorMap, CUtensorMap, TcParams);

template <int NP>
TcKernel pick_np(bool perch, bool comp) {
  if (perch) return comp ? decode_tc_kernel<NP, true, true> : decode_tc_kernel<NP, true, false>;
  return comp ? decode_tc_kernel<NP, false, true> : decode_tc_kernel<NP, false, false>;
}

TcKernel pick_tc(int NP, bool perch, bool comp) {
  switch (NP) {
    case 16: return pick_np<16>(perch, comp);
    case 32: return pick_np<32>(perch, comp);
    default: return pick_np<64>(perch, comp);
  }
}

int np_for(int M) { return M <= 16 ? 16 : M <= 32 ? 32 : 64; }

// ---------------------------------------------------------------- plan --
struct TcPlan {
  int device, N, K, G, rank, comp, NP, gh;     // key
  int S, RT, tiles, units, BF;
  size_t smem;
  uint32_t off_bf, off_x16, off_xr, off_B;
  size_t off_sync, off_P, off_T, total;
  TcKernel fn;
};

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

size_t tile_smem(int NP, int BF, int nr_max, int rank, TcPlan* c) {
  size_t off = (size_t)kRawStages * kRawBytes;
  c->off_bf = (uint32_t)off;
  off += (size_t)BF * kBfBytes;
  c->off_x16 = (uint32_t)off;
  off += (size_t)kX16Stages * kX16Bytes;
  c->off_xr = (uint32_t)off;
  off += (size_t)kXrStages * NP * 128;
  c->off_B = (uint32_t)off;
  off += (size_t)align_up(nr_max, 16) * (2 * std::max(rank, 8) + 16);   // whole 16-row MMA tiles
  return align_up(off, 1024) + 1024;            // + alignment slack of the dynamic base
}

int build_tc_plan(const spear_w4_layer& L, int NP, bool comp, const DeviceInfo& di, TcPlan* pl) {
  const bool has_rank = L.rank > 0;             // the split depends on this, not on comp_enabled
  const bool perch = L.group_size == L.K;
  pl->NP = NP;
  pl->tiles = (L.N + kTileRows - 1) / kTileRows;
  pl->units = (L.K + kUnitK - 1) / kUnitK;
  pl->RT = has_rank ? (L.rank + 1 + 15) / 16 : 0;
  pl->fn = pick_tc(NP, perch, comp);

  // Producer smem: [NW][MT][4][32] + [16][NP] floats
  // (the last producer then forms T over the same bytes: t [NP][r], the gate
  // logits, the vector gate's weights and hidden units)
  const int gh = comp ? L.gate_hidden : 0;
  const size_t form_T_floats = (size_t)NP * (L.rank + 1) + (gh > 0 ? gate_smem_floats(L.rank, gh) + NP * gate_hid_stride(gh) : 0);
  const size_t prod_smem = std::max(((size_t)(kThreads / 32) * (NP / 8) * 128 + 16 * NP), form_T_floats) * 4 + 1024;
  // the dynamic shared memory a CTA may take next to the kernel's static arrays
  cudaFuncAttributes fa{};
  if (cudaFuncGetAttributes(&fa, pl->fn) != cudaSuccess) return fail(SPEAR_ERR_CUDA, "decode: cudaFuncGetAttributes failed");
  const size_t smem_limit = di.smem_optin > fa.sharedSizeBytes ? di.smem_optin - fa.sharedSizeBytes : 0;

  int best_cost = INT32_MAX;
  TcPlan best{};
  bool found = false;
  for (int S = 1; S <= std::min(kMaxS, pl->units); ++S) {
    TcPlan c = *pl;
    c.S = S;
    // most 128-k halves one CTA takes (a split unit, see TcUnits, counts one)
    const int ub = pl->units / S, uq = pl->units % S;
    const int halves_per = 2 * ub + (uq == 0 ? 0 : (2 * uq <= S && L.K % kUnitK == 0) ? 1 : 2);
    // one producer cluster per 16-row tile of [A; w_g], its S CTAs splitting
    // K: splitting K further over more clusters shortens the producers' loop
    // but takes SMs from the tile clusters, and a larger S (fewer K steps per
    // tile CTA) pays more -- measured at 64 tokens on 4096 x 11008 and
    // 11008 x 4096: 34.1 -> 28.5 us and 45.0 -> 35.3 us per call
    const int nr_max = (kTileRows + S - 1) / S;
    // three fp16 weight steps in flight when they fit, else two
    c.BF = kMaxBfStages;
    size_t sm = tile_smem(NP, c.BF, nr_max, L.rank, &c);
    if (sm > smem_limit) {
      c.BF = 2;
      sm = tile_smem(NP, c.BF, nr_max, L.rank, &c);
    }
    c.smem = std::max(sm, prod_smem);
    if (c.smem > smem_limit) continue;
    // all of the unified L1 / shared-memory array as shared memory (one CTA
    // per SM holds up to ~220 KB of rings)
    if (int rc = ensure_smem_limit(reinterpret_cast<const void*>(c.fn), c.smem)) return rc;
    if (cudaFuncSetAttribute(c.fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared) != cudaSuccess)
      return fail(SPEAR_ERR_CUDA, "decode: cudaFuncSetAttribute failed");
    const int clusters = pl->tiles + c.RT;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(clusters * S);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = c.smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int max_clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&max_clusters, c.fn, &cfg) != cudaSuccess) {
      cudaGetLastError();
      continue;
    }
    if (log_plans()) {
      int per_sm = 0, smem_sm = 0, regs_sm = 0;
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, c.fn, kThreads, c.smem);
      cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, di.device);
      cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, di.device);
      cudaFuncAttributes fa{};
      cudaFuncGetAttributes(&fa, c.fn);
      fprintf(stderr, "[spear]   NP=%d S=%d: smem=%zu blocks/SM=%d max clusters=%d needed=%d | regs=%d static=%zu "
              "local=%zu maxthr=%d carveout=%d | SM smem=%d regs=%d\n", NP, S, c.smem, per_sm, max_clusters,
              clusters, fa.numRegs, fa.sharedSizeBytes, fa.localSizeBytes, fa.maxThreadsPerBlock,
              fa.preferredShmemCarveout, smem_sm, regs_sm);
    }
    if (clusters > max_clusters) continue;       // every CTA must be resident at once
    const int cost = halves_per;
    if (cost < best_cost) {
      best_cost = cost;
      best = c;
      found = true;
    }
  }
  if (!found) return fail(SPEAR_ERR_UNSUPPORTED, "decode: no resident cluster configuration for N=%d K=%d", L.N, L.K);
  *pl = best;

  size_t off = 0;
  pl->off_sync = off; off = align_up(off + 3 * sizeof(unsigned), 256);
  pl->off_P = off;    off = align_up(off + (size_t)NP * (std::max(L.rank, 1) + 4) * 4, 256);
  pl->off_T = off;    off = align_up(off + (size_t)NP * std::max(L.rank, 1) * 4, 256);
  pl->total = off;
  return SPEAR_OK;
}

int get_tc_plan(const spear_w4_layer& L, int M, TcPlan* out) {
  DeviceInfo di;
  if (int rc = device_info(&di)) return rc;
  const int NP = np_for(M);
  const int comp = (L.comp_enabled && L.rank > 0) ? 1 : 0;
  const int gh = comp ? L.gate_hidden : 0;     // the last producer's shared memory holds the vector gate
  static std::mutex mu;
  static std::vector<TcPlan> cache;
  std::lock_guard<std::mutex> lk(mu);
  for (const TcPlan& p : cache)
    if (p.device == di.device && p.N == L.N && p.K == L.K && p.G == L.group_size && p.rank == L.rank &&
        p.comp == comp && p.NP == NP && p.gh == gh) {
      *out = p;
      return SPEAR_OK;
    }
  TcPlan p{};
  if (int rc = build_tc_plan(L, NP, comp != 0, di, &p)) return rc;
  if (log_plans())
    fprintf(stderr, "[spear] decode tc plan N=%d K=%d G=%d rank=%d comp=%d NP=%d: S=%d RT=%d tiles=%d "
            "units=%d BF=%d smem=%zu grid=%d\n", L.N, L.K, L.group_size, L.rank, comp, NP, p.S, p.RT,
            p.tiles, p.units, p.BF, p.smem, (p.tiles + p.RT) * p.S);
  p.device = di.device; p.N = L.N; p.K = L.K; p.G = L.group_size; p.rank = L.rank; p.comp = comp; p.gh = gh;
  if (cache.size() > 4096) cache.clear();
  cache.push_back(p);
  *out = p;
  return SPEAR_OK;
}

}  // namespace

int decode_tc_workspace_bytes(const spear_w4_layer& L, int M, size_t* bytes) {
  TcPlan pl;
  if (int rc = get_tc_plan(L, M, &pl)) return rc;
  *bytes = pl.total;
  return SPEAR_OK;
}

size_t decode_tc_sync_bytes() { return 256; }

int launch_decode_tc(const spear_w4_layer& L, const uint16_t* x, int M, void* y, int out_f32, void* ws,
                     size_t ws_bytes, cudaStream_t st, bool overlap) {
  TcPlan pl;
  if (int rc = get_tc_plan(L, M, &pl)) return rc;
  if (!ws || ws_bytes < pl.total)
    return fail(SPEAR_ERR_WORKSPACE, "decode: workspace of %zu B is smaller than the %zu B needed", ws_bytes, pl.total);
  if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0)
    return fail(SPEAR_ERR_INVALID_ARG, "decode: workspace must be 256-byte aligned");
  CUtensorMap tm_w, tm_x;
  if (int rc = make_tmap(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, L.qweight, L.K / 2, L.N, kUnitK / 2, kTileRows,
                         CU_TENSOR_MAP_SWIZZLE_128B)) return rc;
  if (int rc = make_tmap(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, L.K, M, kStepK, pl.NP,
                         CU_TENSOR_MAP_SWIZZLE_128B)) return rc;
  TcParams p{};
  p.N = L.N; p.K = L.K; p.M = M; p.ng = L.K / L.group_size; p.sym = L.symmetric;
  p.qweight = L.qweight;
  p.S = pl.S; p.RT = pl.RT; p.units = pl.units; p.bf_stages = pl.BF;
  p.r = pl.comp ? L.rank : 0;
  p.n_consumers = pl.tiles * pl.S;
  p.scales = reinterpret_cast<const __half*>(L.scales);
  p.zeros = L.zeros;
  p.x = reinterpret_cast<const __nv_bfloat16*>(x);
  p.y = y; p.out_f32 = out_f32;
  p.A = reinterpret_cast<const __nv_bfloat16*>(L.A);
  p.B = reinterpret_cast<const __nv_bfloat16*>(L.B);
  p.w_g = reinterpret_cast<const __nv_bfloat16*>(L.w_g);
  p.b_g = L.b_g; p.alpha = L.alpha;
  p.gh = L.gate_hidden; p.gw1 = L.gate_w1; p.gc1 = L.gate_c1; p.gw2 = L.gate_w2; p.gc2 = L.gate_c2;
  char* base = reinterpret_cast<char*>(ws);
  p.ws_sync = reinterpret_cast<unsigned*>(base + pl.off_sync);
  p.ws_P = reinterpret_cast<float*>(base + pl.off_P);
  p.ws_T = reinterpret_cast<uint4*>(base + pl.off_T);
  p.t_wait_ns = wait_limit_ns(kTWaitNs);
  p.off_bf = pl.off_bf; p.off_x16 = pl.off_x16; p.off_xr = pl.off_xr; p.off_B = pl.off_B;

  if (int rc = ensure_smem_limit(reinterpret_cast<const void*>(pl.fn), pl.smem)) return rc;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((pl.tiles + pl.RT) * pl.S);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = pl.S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 2 : 1;
  return cuda_check(cudaLaunchKernelEx(&cfg, pl.fn, tm_w, tm_x, p), "decode launch");
}

int read_and_clear_status_decode_tc(unsigned* out, cudaStream_t st) {
  void* addr = nullptr;
  if (int rc = cuda_check(cudaGetSymbolAddress(&addr, g_dtc_status), "decode status address")) return rc;
  if (int rc = cuda_check(cudaMemcpyAsync(out, addr, sizeof(unsigned), cudaMemcpyDeviceToHost, st),
                          "read decode status")) return rc;
  if (int rc = cuda_check(cudaStreamSynchronize(st), "read decode status")) return rc;
  return cuda_check(cudaMemsetAsync(addr, 0, sizeof(unsigned), st), "clear decode status");
}

}  // namespace spear
