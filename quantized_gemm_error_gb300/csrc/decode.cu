// decode.cu -- fused decode kernel for the gated W4 + low-rank compensated
// linear (SPEAR explainer, Technical Summary 2.2 A: in the memory-bound decode
// phase the compensator is fused into the low-bit GEMM epilogue so the layer
// is ONE kernel launch).
//
//   y[m][n] = sum_k (u[n][k] - z[n][g]) s[n][g] x[m][k]  +  alpha g_m sum_j B[n][j] t_m[j]
//   t_m = A x_m,  g_m = sigmoid(w_g . x_m + b_g)
//
// Design (one launch; the plan keeps every block resident at once, and the
// producers, which wait for nothing, have the lowest block indices):
//  * Producer blocks (the first Q) compute the rank-(r+1) down-projection
//    P = [A; w_g] x over disjoint K slices with bf16 mma.sync, write their
//    slice partials to the workspace, and the last producer to arrive sums
//    them in a fixed order, applies the gate and publishes T = alpha g t with
//    a release flag.
//  * Streamer blocks own contiguous ranges of whole 16-row tiles of the int4
//    weight (tile counts per block differ by at most one), so no partial sum
//    leaves a block; the block's 8 warps split each tile's K range.  Weights
//    move global -> shared through a per-warp cp.async ring (L1 bypass), are
//    turned into exact small integers in registers (nibble | bf16 bias, minus
//    the biased zero point) and multiplied by the tokens with mma.sync; the
//    group scale is applied to each 128-k partial in fp32.
//  * Only the epilogue depends on T.  A helper warp of each streamer block
//    stages the block's factor-B rows, waits (bounded) for the flag, loads T
//    into shared memory while the other eight warps stream the weights, and
//    hands both over at one named barrier before the epilogue, which adds B T
//    with one more small mma and stores y.  The last helper past the flag
//    resets it, so the workspace's synchronisation words are zero again
//    between calls.
//
// HBM traffic per call: N K / 2 (codes) + N K/G * 2 (scales) + zeros + (r+1) K 2
// (A, w_g) + N r 2 (B) + M K 2 (x) + M N 2 (y): the roofline of this kernel.
#include <algorithm>
#include <cstdio>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace spear {
namespace {

__device__ unsigned g_decode_status;

using sm100::named_arrive;
using sm100::named_sync;

constexpr int kThreads = 256;              // the warps that compute
constexpr int kWarps = 8;
constexpr int kBlockThreads = kThreads + 32; // + one helper warp (streamer blocks of compensated layers)
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
  int gh;                   // vector-gate hidden width (0: the scalar gate)
  const float *gw1, *gc1, *gw2, *gc2;
  // work split
  int Q, P;                 // producer / streamer blocks
  int tiles, nchunks;       // N/16, K/128
  int max_tiles;            // most tiles one streamer owns
  int ng;                   // K/G
  // workspace
  float* ws_prod;           // [Q][Mpad][16]
  float* ws_T;              // [Mpad][r]
  unsigned* ws_sync;        // [0] producer ticket, [1] T flag, [2] streamer ticket
  uint64_t wait_ns;         // limit of the wait for T
  size_t smem_bytes;        // dynamic shared memory of the launch (index checks of the debug build)
};


// ---------------------------------------------------------------- producer --
// Producer block q computes the partial P[m][i] = sum_{k in slice s} W'[i][k] x[m][k]
// for one 16-row tile rt = q % RT of W' = [A; w_g; 0-padding] over K slice
// s = q / RT (S = Q / RT slices), so its loads take one round trip.
// Lane (g, c) of a warp loads 16 B (8 consecutive k) per row; within a 32-k
// piece the MMA's k positions {2c, 2c+1, 2c+8, 2c+9} of k-step h map to the
// lane's k = 8c + 4h + {0, 1, 2, 3}, identically for both operands.
constexpr int kMaxSlices = 16;
// producer scratch: cross-warp sums (t and the hidden units reuse them), then
// the staged gate weights; the streamers' ring alone is larger
static_assert(kWarps * 2 * 128 >= 16 * (64 + gate_hid_stride(32)), "t and hidden units fit over the cross-warp sums");
static_assert(kWarps * kStages * 2 * 32 * 16 >= (kWarps * 2 * 128 + gate_smem_floats(64, 32)) * 4,
              "producer scratch within the streamer's shared memory");

template <int MT>
__device__ void producer_block(const DecodeParams& p, float* smem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int RT = (p.r + 1 + 15) / 16;
  const int Mpad = MT * 8;
  const int q = blockIdx.x, rt = q % RT, sl = q / RT, S = p.Q / RT;
  const int c0 = (int)((long long)sl * p.nchunks / S), c1 = (int)((long long)(sl + 1) * p.nchunks / S);
  const int npieces = (c1 - c0) * 4;                   // 32-k pieces of the slice
  SPEAR_CHECK(&g_decode_status, 0 <= c0 && c0 <= c1 && c1 <= p.nchunks && sl < S && S <= kMaxSlices);
  float* red = smem;                                   // [kWarps][MT][4][32]
  // the vector gate's weights, copied while the slice streams (every producer:
  // which one sums the slices is known only at the end)
  float* gs = smem + kWarps * MT * 128;                // W1 [h][r], W2 [r][h], c1 [h], c2 [r]
  if (p.gh > 0) stage_gate_weights_async(p.gw1, p.gw2, p.gc1, p.gc2, p.r, p.gh, gs, threadIdx.x, kThreads);

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
  // U pieces per pass: all of their loads are in flight together (the plan
  // sizes the slices so that one pass covers a warp's share)
  constexpr int U = MT == 1 ? 4 : MT == 2 ? 2 : 1;
  // the rows of A and w_g are weights: the first pass loads them before
  // waiting for the kernel ahead (overlapped launches), then the tokens
  bool waited = false;
  for (int pc0 = warp; pc0 < npieces; pc0 += U * kWarps) {
    uint4 va[U], vb[U], xv[U][MT];
#pragma unroll
    for (int h = 0; h < U; ++h) {
      const int pc = pc0 + h * kWarps;
      const bool ok = pc < npieces;
      const int kb = c0 * kChunkK + pc * 32 + 8 * c;
      va[h] = (ok && wlo) ? ldg16(wlo + kb) : make_uint4(0, 0, 0, 0);
      vb[h] = (ok && whi) ? ldg16(whi + kb) : make_uint4(0, 0, 0, 0);
    }
    if (!waited) {
      pdl_wait();
      waited = true;
    }
#pragma unroll
    for (int h = 0; h < U; ++h) {
      const int pc = pc0 + h * kWarps;
      const bool ok = pc < npieces;
      const int kb = c0 * kChunkK + pc * 32 + 8 * c;
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
  if (p.gh > 0) cp_async_wait<0>();                        // the gate weights (published by the barrier below)
  // cross-warp sum in a fixed order; this block's partial for its 16 rows
#pragma unroll
  for (int t = 0; t < MT; ++t)
#pragma unroll
    for (int i = 0; i < 4; ++i) red[((warp * MT + t) * 4 + i) * 32 + lane] = acc[t][i];
  named_sync(1, kThreads);
  for (int e = threadIdx.x; e < MT * 4 * 32; e += kThreads) {
    const int t = e / 128, i = (e / 32) & 3, ln = e & 31;
    float v = 0.0f;
    for (int w = 0; w < kWarps; ++w) v += red[((w * MT + t) * 4 + i) * 32 + ln];
    // C fragment element i of lane ln: row (ln/4) + 8 (i/2), token t*8 + 2 (ln%4) + (i%2)
    const int row = (ln >> 2) + 8 * (i >> 1);
    const int tok = t * 8 + 2 * (ln & 3) + (i & 1);
    SPEAR_CHECK(&g_decode_status, q < p.Q && tok < Mpad && row < 16);
    p.ws_prod[((size_t)q * Mpad + tok) * 16 + row] = v;
  }
  named_sync(1, kThreads);

  // arrive; the last producer sums the slices, applies the gate, publishes T.
  // The ticket is an acquire-release atomic: it publishes this block's
  // partials (ordered before it by the barrier) and, in the last producer,
  // makes every other producer's partials visible.
  __shared__ unsigned s_last;
  if (threadIdx.x == 0) {
    const unsigned old = atom_add_acq_rel_gpu(&p.ws_sync[0], 1u);
    s_last = (old == (unsigned)(p.Q - 1));
  }
  named_sync(1, kThreads);
  if (!s_last) return;
  auto slice_sum = [&](int m, int i) {                  // fixed order over slices
    const int rti = i / 16, ri = i % 16;
    float part[kMaxSlices];
#pragma unroll
    SPEAR_CHECK(&g_decode_status, (S - 1) * RT + rti < p.Q && m < Mpad);
    for (int ss = 0; ss < kMaxSlices; ++ss)
      part[ss] = ss < S ? __ldcg(p.ws_prod + ((size_t)(ss * RT + rti) * Mpad + m) * 16 + ri) : 0.0f;
    float v = 0.0f;
#pragma unroll
    for (int ss = 0; ss < kMaxSlices; ++ss) v += part[ss];
    return v;
  };
  if (p.gh > 0) {
    // vector gate: t [Mpad][r] into shared memory, then one warp per token
    // forms gamma(t) and T = alpha gamma(t) t
    float* ts = smem;                                   // [Mpad][r] (over the spent cross-warp sums)
    float* hs = ts + Mpad * p.r;                        // [Mpad][h | 1] hidden units
    const GateSmem gt(gs, p.r, p.gh);
    for (int e = threadIdx.x; e < Mpad * p.r; e += kThreads) ts[e] = slice_sum(e / p.r, e % p.r);
    named_sync(1, kThreads);
    vector_gate_hidden_rows(ts, Mpad, gt, hs, threadIdx.x, kThreads);
    named_sync(1, kThreads);
    vector_gate_apply_rows(ts, Mpad, gt, hs, threadIdx.x, kThreads);
    named_sync(1, kThreads);
    for (int e = threadIdx.x; e < Mpad * p.r; e += kThreads)
      p.ws_T[e] = (e / p.r < p.M) ? p.alpha * ts[e] : 0.0f;
  } else {
    // t and the gate row in one pass over the slices, then T = alpha g t
    float* ts = smem;                                   // [Mpad][r + 1] (over the spent cross-warp sums)
    const int rr = p.r + 1;
    for (int e = threadIdx.x; e < Mpad * rr; e += kThreads) ts[e] = slice_sum(e / rr, e % rr);
    named_sync(1, kThreads);
    for (int e = threadIdx.x; e < Mpad * p.r; e += kThreads) {
      const int m = e / p.r, j = e % p.r;
      const float gate = 1.0f / (1.0f + expf(-(ts[m * rr + p.r] + p.b_g)));
      p.ws_T[e] = (m < p.M) ? p.alpha * gate * ts[m * rr + j] : 0.0f;
    }
  }
  // T is published by thread 0's release store, ordered after every
  // thread's T writes by the barrier
  named_sync(1, kThreads);
  if (threadIdx.x == 0) {
    p.ws_sync[0] = 0;                                   // ticket ready for the next call
    st_release_gpu(&p.ws_sync[1], 1u);
  }
}

// ---------------------------------------------------------------- streamer --
// Block b owns whole 16-row tiles [t0, t1) of Wq (t = b * tiles / P), so no
// partial sum ever leaves the block.  Its 8 warps split each tile's K range
// (warp w takes chunks w, w + 8, ...); weights stream through a per-warp
// cp.async ring in the order (tile, chunk) and become exact small integers in
// registers; the tokens enter mma.sync as B fragments.
//
// XS (M <= 8, tokens small enough for shared memory): the block first copies x
// as fp16 (exact for |x| < 65504) in B-fragment order and keeps per-128-k sums
// of the even-k and odd-k tokens.  The weights then enter fp16 MMAs straight
// from the nibbles with no subtraction -- the low nibble of each byte becomes
// 1024 + u through an fp16 exponent bias, the high nibble (left in place)
// 64 + u -- and the constant parts and the zero point are removed per 128-k
// chunk in fp32:
//   sum_k (u_k - z) x_k = sum_k (c_k + u_k) x_k - (1024 + z) E - (64 + z) O,
//   c_k = 1024 (k even) or 64 (k odd),  E / O = sums of x over even / odd k.
// Otherwise the nibbles become 128 + u through a bf16 bias, the biased zero
// point is subtracted (exact), and bf16 MMAs read the tokens from L1.
template <int MT, bool COMP, bool PERCH, bool XS>
__device__ void streamer_block(const DecodeParams& p, float* smem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int b = blockIdx.x - p.Q;
  const int t0 = (int)((long long)b * p.tiles / p.P), t1 = (int)((long long)(b + 1) * p.tiles / p.P);
  const int ntl = t1 - t0;                                   // tiles of this block
  const int Mpad = MT * 8;
  const size_t half_k = (size_t)p.K / 2;
  const int k8 = p.K / 8;
  const int xrow = k8 + 1;

  uint4* ring = reinterpret_cast<uint4*>(smem);                       // [kWarps][kStages][2][32]
  float* red = smem + kWarps * kStages * 2 * 32 * 4;                  // [kWarps][MT][4][32]
  float* ybuf = red + kWarps * MT * 4 * 32;                           // [max_tiles][MT][4][32]
  uint32_t* Ts = reinterpret_cast<uint32_t*>(ybuf + p.max_tiles * MT * 4 * 32);  // [Mpad][r/2] hi, then lo
  // the block's rows of scales, zero-point bytes and factor B, as laid out
  // in global memory (each a contiguous range: whole 16-row tiles)
  __half* sc_s = reinterpret_cast<__half*>(Ts + (COMP ? Mpad * kMaxRank : 0));   // [max_tiles * 16][ng]
  uint8_t* z_s = reinterpret_cast<uint8_t*>(sc_s + p.max_tiles * 16 * p.ng);     // [max_tiles * 16][zrow]
  const int zrow = (p.ng + 1) / 2;
  __nv_bfloat16* B_s = reinterpret_cast<__nv_bfloat16*>(smem_align_up(z_s + p.max_tiles * 16 * zrow, 16));  // [max_tiles * 16][r]
  uint4* xs = reinterpret_cast<uint4*>(
      smem_align_up(reinterpret_cast<uint8_t*>(B_s + (COMP ? p.max_tiles * 16 * p.r : 0)), 16));   // [M][xrow] (XS)
  float* Ps = reinterpret_cast<float*>(xs + (XS ? p.M * xrow : 0));  // [M][nchunks] 1024 E + 64 O (XS)
  float* Xs = Ps + (XS ? p.M * p.nchunks : 0);                       // [M][nchunks] E + O (XS)
  __shared__ int s_xbigw[kWarps];                          // per compute warp: a staged unit reaches 2^15 (rare)
  __shared__ unsigned s_xmax[8];                           // bits of max |x| per staged token (rare path)
  __shared__ float s_xdn[8], s_xup[8];                     // 2^-e, 2^e per staged token
  SPEAR_CHECK(&g_decode_status, 0 <= t0 && t0 <= t1 && t1 <= p.tiles && ntl <= p.max_tiles);
  SPEAR_CHECK(&g_decode_status, reinterpret_cast<const uint8_t*>(Xs + (XS ? p.M * p.nchunks : 0)) <=
                                    reinterpret_cast<const uint8_t*>(smem) + p.smem_bytes);

  if (warp == kWarps) {
    // ------------------------------------------------ helper warp
    // The factor-B rows (weights: before waiting for the kernel ahead), then
    // the flag (bounded), a ticket, and T as bf16 hi + lo (T = hi + lo to
    // ~2^-16 relative), all while the compute warps stream the weights.
    if (!COMP) return;
    const size_t row0 = (size_t)t0 * 16, nb = (size_t)ntl * 16 * p.r * 2 / 16;
    for (size_t e = lane; e < nb; e += 32)
      cp_async16(reinterpret_cast<uint4*>(B_s) + e, reinterpret_cast<const uint4*>(p.B + row0 * p.r) + e);
    cp_async_commit();
    pdl_wait();                                             // the workspace follows the kernel ahead
    unsigned ok = 0, ticket = 0;
    if (lane == 0) {
      const uint64_t tw = globaltimer_ns();
      for (unsigned i = 0;; ++i) {
        if (ld_acquire_gpu(&p.ws_sync[1])) { ok = 1; break; }
        if ((i & 63) == 63 && globaltimer_ns() - tw > p.wait_ns) break;
        __nanosleep(32);
      }
      if (!ok) record_status(&g_decode_status, DEV_ERR_TIMEOUT);
      ticket = atomicAdd(&p.ws_sync[2], 1u);
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    // all of this lane's pairs of T in flight at once (one L2 round trip)
    constexpr int kTPairs = MT * 8 * kMaxRank / 2 / 32;
    const int npairs = Mpad * p.r / 2;
    SPEAR_CHECK(&g_decode_status, 2 * npairs <= Mpad * kMaxRank && p.r <= kMaxRank);
    float2 tv[kTPairs];
#pragma unroll
    for (int i = 0; i < kTPairs; ++i) {
      const int e = lane + 32 * i;
      tv[i] = (ok && e < npairs) ? __ldcg(reinterpret_cast<const float2*>(p.ws_T) + e) : make_float2(0.0f, 0.0f);
    }
#pragma unroll
    for (int i = 0; i < kTPairs; ++i) {
      const int e = lane + 32 * i;                          // pair e: T[m][2 jj'], T[m][2 jj' + 1]
      if (e < npairs) {
        const __nv_bfloat16 h0 = __float2bfloat16_rn(tv[i].x), h1 = __float2bfloat16_rn(tv[i].y);
        Ts[e] = pack_bf16x2(__bfloat162float(h0), __bfloat162float(h1));
        Ts[npairs + e] = pack_bf16x2(tv[i].x - __bfloat162float(h0), tv[i].y - __bfloat162float(h1));
      }
    }
    cp_async_wait<0>();                                     // the B rows
    named_arrive(2, kBlockThreads);                         // B rows and T are in place
    if (lane == 0 && ticket == (unsigned)(p.P - 1)) {       // every streamer is past its wait
      p.ws_sync[2] = 0;
      atomicExch(&p.ws_sync[1], 0u);
    }
    return;
  }

  // work items of this warp: (tile, chunk), chunk = warp + 8 j; the issue
  // cursor walks them with pointer increments only
  const int per_tile = (p.nchunks - warp + kWarps - 1) / kWarps;     // chunks of each tile for this warp
  const int nitems = ntl * per_tile;
  uint4* my_ring = ring + warp * kStages * 2 * 32;
  const uint8_t* tile_base = p.qweight + (size_t)(t0 * 16 + g) * half_k + (size_t)warp * (kChunkK / 2) + c * 16;
  const size_t tile_step = 16 * half_k;                              // bytes between tiles
  const uint8_t* src = tile_base;
  int issued = 0, ij = 0;
  auto issue = [&](int slot) {
    if (issued < nitems) {
      SPEAR_CHECK(&g_decode_status, slot < kStages && src >= p.qweight &&
                                        src + 8 * half_k + 16 <= p.qweight + (size_t)p.N * half_k);
      cp_async16(my_ring + (slot * 2 + 0) * 32 + lane, src);
      cp_async16(my_ring + (slot * 2 + 1) * 32 + lane, src + 8 * half_k);
      ++issued;
      if (++ij == per_tile) { ij = 0; tile_base += tile_step; src = tile_base; }
      else src += kWarps * (kChunkK / 2);
    }
    cp_async_commit();
  };

  // 1. tokens (XS) into registers (they come from L2); then, as one cp.async
  // group ahead of the weight stream, the block's scales and zero points, so
  // the only wait before the main loop is for bytes that travel together with
  // the first weights
  const int xunits = XS ? p.M * k8 : 0;
  constexpr int kXBatch = XS ? 4 : 1;
  uint4 xr[kXBatch];
  {
    auto stage = [&](void* dst, const void* src_base, size_t bytes) {
      for (size_t e = threadIdx.x; e < bytes / 16; e += kThreads)
        cp_async16(reinterpret_cast<uint4*>(dst) + e, reinterpret_cast<const uint4*>(src_base) + e);
    };
    const size_t row0 = (size_t)t0 * 16, rows = (size_t)ntl * 16;
    stage(sc_s, p.scales + row0 * p.ng, rows * p.ng * 2);
    if (!p.sym) stage(z_s, p.zeros + row0 * zrow, rows * zrow);
    cp_async_commit();
  }
#pragma unroll
  for (int st = 0; st < kStages - 1; ++st) issue(st);
  // everything above reads only the layer's weights; x, the workspace and y
  // may belong to the kernel before this one (overlapped launches)
  pdl_wait();
  if (XS) {
#pragma unroll
    for (int j = 0; j < kXBatch; ++j) {
      const int e = threadIdx.x + j * kThreads;
      xr[j] = e < xunits ? ldg16(p.x + (size_t)e * 8) : make_uint4(0, 0, 0, 0);
    }
  }
  if (!XS) {
    // token rows of this warp's first two chunks into L1 (16 tokens x 256 B per chunk)
    for (int jj = 0; jj < 2 && jj < per_tile; ++jj) {
      const int ch = warp + kWarps * jj;
      for (int q = lane; q < Mpad * 2; q += 32) {
        const int tok = q >> 1;
        if (tok < p.M) prefetch_l1(p.x + (size_t)tok * p.K + ch * kChunkK + (q & 1) * 64);
      }
    }
  }

  // 2. tokens for XS: fp16 in B-fragment order plus per-chunk even/odd sums.
  // A token whose max |x| reaches 2^15 enters as x 2^-e (power-of-two token
  // scaling: exact in fp16 down to 2^-24 2^e); the epilogue multiplies its
  // outputs by 2^e.  The pass below converts every token unscaled and only
  // flags a value at or above 2^15 (or not finite); the (rare) flagged call
  // then takes each token's maximum and converts the tokens that need it again.
  bool any_big = false;
  if (XS) {
    bool big = false;
    // 16 consecutive units (128 k) of one token are 16 consecutive lanes: their
    // E / O partials and maxima reduce with 4 shuffles (padding units contribute zeros).
    auto stage = [&](int e, uint4 v, float sc, bool write) -> float {
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};            // (x0,x1) (x2,x3) (x4,x5) (x6,x7)
      float f[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) { f[2 * i] = bf16x2_lo(w[i]) * sc; f[2 * i + 1] = bf16x2_hi(w[i]) * sc; }
      float ev = (f[0] + f[2]) + (f[4] + f[6]);
      float od = (f[1] + f[3]) + (f[5] + f[7]);
#pragma unroll
      for (int i = 0; i < 8; ++i) big |= !(fabsf(f[i]) < 32768.0f);
      auto h2 = [](float lo, float hi) {
        const __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
      };
      if (write && e < xunits) {
        const int m = e / k8, kk = e % k8;
        xs[m * xrow + kk] = make_uint4(h2(f[0], f[4]), h2(f[1], f[5]), h2(f[2], f[6]), h2(f[3], f[7]));
      }
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) {
        ev += __shfl_xor_sync(0xffffffffu, ev, o);
        od += __shfl_xor_sync(0xffffffffu, od, o);
      }
      if (write && (lane & 15) == 0 && e < xunits) {
        const int m = e / k8, ch = (e % k8) / 16;
        Ps[m * p.nchunks + ch] = 1024.0f * ev + 64.0f * od;
        Xs[m * p.nchunks + ch] = ev + od;
      }
    };
    for (int j0 = 0; j0 < xunits; j0 += kThreads * kXBatch) {
#pragma unroll
      for (int j = 0; j < kXBatch; ++j) {
        const int e = threadIdx.x + j0 + j * kThreads;
        uint4 v;
        if (j0 == 0) v = xr[j];
        else v = e < xunits ? ldg16(p.x + (size_t)e * 8) : make_uint4(0, 0, 0, 0);
        stage(e, v, 1.0f, true);
      }
    }
    big = __any_sync(0xffffffffu, big);
    if (lane == 0) s_xbigw[warp] = big ? 1 : 0;            // read after the barrier below
  }
  cp_async_wait<kStages - 1>();                            // the staged scales, zeros and B
  named_sync(1, kThreads);
  if (XS) {
#pragma unroll
    for (int w = 0; w < kWarps; ++w) any_big |= s_xbigw[w] != 0;
  }
  if (XS && any_big) {
    // rare: each token's max |x|, its scale, and the tokens at or above 2^15
    // converted again with it (E / O sums too); a non-finite value is reported
    if (threadIdx.x < 8) s_xmax[threadIdx.x] = 0u;
    named_sync(1, kThreads);
    for (int e0 = 0; e0 < xunits; e0 += kThreads) {
      const int e = threadIdx.x + e0;
      float amax = e < xunits ? bf16x8_absmax(ldg16(p.x + (size_t)e * 8)) : 0.0f;
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      if ((lane & 15) == 0 && e < xunits) atomicMax(&s_xmax[e / k8], __float_as_uint(amax));
    }
    named_sync(1, kThreads);
    if (threadIdx.x < 8) {
      const int ex = token_scale_exp(__uint_as_float(s_xmax[threadIdx.x]));
      s_xdn[threadIdx.x] = exp2_int(-ex);
      s_xup[threadIdx.x] = exp2_int(ex);
    }
    named_sync(1, kThreads);
    bool bad = false;
    for (int e0 = 0; e0 < xunits; e0 += kThreads) {
      const int e = threadIdx.x + e0;
      const int m = e < xunits ? e / k8 : 0;
      const uint4 v = e < xunits ? ldg16(p.x + (size_t)e * 8) : make_uint4(0, 0, 0, 0);
      // (the same per-unit work as the first pass, for the tokens with a scale)
      const float sc = s_xdn[m];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      float f[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) { f[2 * i] = bf16x2_lo(w[i]) * sc; f[2 * i + 1] = bf16x2_hi(w[i]) * sc; }
      float ev = (f[0] + f[2]) + (f[4] + f[6]);
      float od = (f[1] + f[3]) + (f[5] + f[7]);
      bad |= !(bf16x8_absmax(v) <= 3.4e38f);
      const bool write = e < xunits && s_xup[m] != 1.0f;
      if (write) {
        auto h2 = [](float lo, float hi) {
          const __half2 h = __floats2half2_rn(lo, hi);
          return *reinterpret_cast<const uint32_t*>(&h);
        };
        xs[m * xrow + e % k8] = make_uint4(h2(f[0], f[4]), h2(f[1], f[5]), h2(f[2], f[6]), h2(f[3], f[7]));
      }
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) {
        ev += __shfl_xor_sync(0xffffffffu, ev, o);
        od += __shfl_xor_sync(0xffffffffu, od, o);
      }
      if (write && (lane & 15) == 0) {
        const int ch = (e % k8) / 16;
        Ps[m * p.nchunks + ch] = 1024.0f * ev + 64.0f * od;
        Xs[m * p.nchunks + ch] = ev + od;
      }
    }
    if (bad) record_status(&g_decode_status, DEV_ERR_INVALID);
    named_sync(1, kThreads);
  }

  // 3. main loop
  int slot = 0;
  const bool tok_ok = g < p.M;
  const int u0 = 2 * c, u1 = 2 * c + 1;                   // this lane's output tokens (XS)
  const bool ok0 = u0 < p.M, ok1 = u1 < p.M;
  for (int tl = 0; tl < ntl; ++tl) {
    float acc[MT][4];
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[t][i] = 0.0f;
    const int srow = tl * 16 * p.ng;
    const __half* sc_lo = sc_s + srow + g * p.ng;
    const __half* sc_hi = sc_lo + 8 * p.ng;
    const uint8_t* z_lo = z_s + (tl * 16 + g) * zrow;
    const uint8_t* z_hi = z_lo + 8 * zrow;
    auto zero_at = [&](const uint8_t* zr, int gi) -> int {
      return p.sym ? 8 : (gi & 1) ? (zr[gi >> 1] >> 4) : (zr[gi >> 1] & 15);
    };
    for (int j = 0; j < per_tile; ++j) {
      issue((slot + kStages - 1) % kStages);
      cp_async_wait<kStages - 1>();
      const int ch = warp + kWarps * j;
      const int gi = PERCH ? 0 : ch;                       // group 128 = one chunk
      const uint4 wlo = my_ring[(slot * 2 + 0) * 32 + lane];
      const uint4 whi = my_ring[(slot * 2 + 1) * 32 + lane];
      const uint32_t wl[4] = {wlo.x, wlo.y, wlo.z, wlo.w};
      const uint32_t wh[4] = {whi.x, whi.y, whi.z, whi.w};
      const int zl = zero_at(z_lo, gi), zh = zero_at(z_hi, gi);
      // two accumulators per token tile (the two k-steps of each 32-k piece)
      // halve the dependent MMA chain
      float part[MT][4], part2[MT][4];
#pragma unroll
      for (int t = 0; t < MT; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) part[t][i] = part2[t][i] = 0.0f;
      if (!XS && j + 2 < per_tile) {
        // token rows of the chunk after next into L1 (16 tokens x 256 B)
        const int chn = warp + kWarps * (j + 2);
        for (int q = lane; q < Mpad * 2; q += 32) {
          const int tok = q >> 1;
          if (tok < p.M) prefetch_l1(p.x + (size_t)tok * p.K + chn * kChunkK + (q & 1) * 64);
        }
      }
      if constexpr (XS) {
        const uint4* xrowp = xs + g * xrow + ch * 16 + 4 * c;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint32_t l8 = wl[w] >> 8, h8 = wh[w] >> 8;
          // step 0: (n0, n4) as 1024 + u, (n1, n5) as 64 + u; step 1: the same for n2 .. n7
          const uint32_t a0 = (wl[w] & 0x000F000Fu) | 0x64006400u, a1 = (wh[w] & 0x000F000Fu) | 0x64006400u;
          const uint32_t a2 = (wl[w] & 0x00F000F0u) | 0x54005400u, a3 = (wh[w] & 0x00F000F0u) | 0x54005400u;
          const uint32_t e0 = (l8 & 0x000F000Fu) | 0x64006400u, e1 = (h8 & 0x000F000Fu) | 0x64006400u;
          const uint32_t e2 = (l8 & 0x00F000F0u) | 0x54005400u, e3 = (h8 & 0x00F000F0u) | 0x54005400u;
          const uint4 xv = tok_ok ? xrowp[w] : make_uint4(0, 0, 0, 0);
          mma_f16_16816(part[0], a0, a1, a2, a3, xv.x, xv.y);
          mma_f16_16816(part2[0], e0, e1, e2, e3, xv.z, xv.w);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) part[0][i] += part2[0][i];
        const float P0 = ok0 ? Ps[u0 * p.nchunks + ch] : 0.0f, X0 = ok0 ? Xs[u0 * p.nchunks + ch] : 0.0f;
        const float P1 = ok1 ? Ps[u1 * p.nchunks + ch] : 0.0f, X1 = ok1 ? Xs[u1 * p.nchunks + ch] : 0.0f;
        part[0][0] -= fmaf((float)zl, X0, P0);
        part[0][1] -= fmaf((float)zl, X1, P1);
        part[0][2] -= fmaf((float)zh, X0, P0);
        part[0][3] -= fmaf((float)zh, X1, P1);
      } else {
        const uint32_t zlo = bf16x2_bias((uint32_t)zl), zhi = bf16x2_bias((uint32_t)zh);
        const size_t kbase = (size_t)ch * kChunkK + 32 * c;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          uint32_t va[4], vb[4];
          nibbles_to_bf16x2_biased(wl[w], va);
          nibbles_to_bf16x2_biased(wh[w], vb);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            va[i] = bf16x2_sub(va[i], zlo);                  // exact (u - z)
            vb[i] = bf16x2_sub(vb[i], zhi);
          }
#pragma unroll
          for (int t = 0; t < MT; ++t) {
            const int tok = t * 8 + g;
            const uint4 xv = tok < p.M ? ldg16(p.x + (size_t)tok * p.K + kbase + 8 * w) : make_uint4(0, 0, 0, 0);
            // k positions: step 0 pairs nibbles (0,4),(1,5); step 1 pairs (2,6),(3,7)
            const uint32_t b00 = __byte_perm(xv.x, xv.z, 0x5410), b01 = __byte_perm(xv.x, xv.z, 0x7632);
            const uint32_t b10 = __byte_perm(xv.y, xv.w, 0x5410), b11 = __byte_perm(xv.y, xv.w, 0x7632);
            mma_bf16_16816(part[t], va[0], vb[0], va[1], vb[1], b00, b01);
            mma_bf16_16816(part2[t], va[2], vb[2], va[3], vb[3], b10, b11);
          }
        }
#pragma unroll
        for (int t = 0; t < MT; ++t)
#pragma unroll
          for (int i = 0; i < 4; ++i) part[t][i] += part2[t][i];
      }
      if (PERCH) {
#pragma unroll
        for (int t = 0; t < MT; ++t)
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[t][i] += part[t][i];
      } else {
        const float slo = __half2float(sc_lo[gi]);
        const float shi = __half2float(sc_hi[gi]);
#pragma unroll
        for (int t = 0; t < MT; ++t) {
          acc[t][0] = fmaf(slo, part[t][0], acc[t][0]);
          acc[t][1] = fmaf(slo, part[t][1], acc[t][1]);
          acc[t][2] = fmaf(shi, part[t][2], acc[t][2]);
          acc[t][3] = fmaf(shi, part[t][3], acc[t][3]);
        }
      }
      slot = (slot + 1) % kStages;
    }
    // tile done: fixed-order sum over the warps
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
      for (int i = 0; i < 4; ++i) red[((warp * MT + t) * 4 + i) * 32 + lane] = acc[t][i];
    named_sync(1, kThreads);
    for (int e = threadIdx.x; e < MT * 128; e += kThreads) {
      float v = 0.0f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) v += red[w * MT * 128 + e];
      ybuf[tl * MT * 128 + e] = v;
    }
    named_sync(1, kThreads);
  }
  cp_async_wait<0>();

  // 4. the compensator's down-projection and the B rows (from the helper warp)
  if (COMP) named_sync(2, kBlockThreads);

  // 5. epilogue: y = acc (* per-channel scale) + B T, one (tile, token tile) per warp
  for (int item = warp; item < ntl * MT; item += kWarps) {
    const int tl = item / MT, t = item % MT;
    const int n_lo = (t0 + tl) * 16 + g, n_hi = n_lo + 8;
    float v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = ybuf[(tl * MT + t) * 128 + i * 32 + lane];
    if (PERCH) {
      const float slo = __half2float(sc_s[tl * 16 * p.ng + g * p.ng]);
      const float shi = __half2float(sc_s[tl * 16 * p.ng + (g + 8) * p.ng]);
      v[0] *= slo; v[1] *= slo; v[2] *= shi; v[3] *= shi;
    }
    if (XS && any_big) {                                   // staged tokens' scale 2^e (outputs of tokens 2c, 2c + 1)
      const float u0 = 2 * c < p.M ? s_xup[2 * c] : 1.0f, u1 = 2 * c + 1 < p.M ? s_xup[2 * c + 1] : 1.0f;
      v[0] *= u0; v[1] *= u1; v[2] *= u0; v[3] *= u1;
    }
    if (COMP) {
      const int rh = p.r / 2;
      for (int j0 = 0; j0 < p.r; j0 += 16) {
        const uint32_t* Blo = reinterpret_cast<const uint32_t*>(B_s + (size_t)(tl * 16 + g) * p.r + j0);
        const uint32_t* Bhi = reinterpret_cast<const uint32_t*>(B_s + (size_t)(tl * 16 + g + 8) * p.r + j0);
        const uint32_t a0 = Blo[c], a1 = Bhi[c], a2 = Blo[c + 4], a3 = Bhi[c + 4];
        const int tok = t * 8 + g;
        const uint32_t* th = Ts + tok * rh + j0 / 2;
        const uint32_t* tlo = Ts + Mpad * rh + tok * rh + j0 / 2;
        mma_bf16_16816(v, a0, a1, a2, a3, th[c], th[c + 4]);
        mma_bf16_16816(v, a0, a1, a2, a3, tlo[c], tlo[c + 4]);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int tok = t * 8 + 2 * c + (i & 1);
      const int n = (i < 2) ? n_lo : n_hi;
      if (tok < p.M) {
        SPEAR_CHECK(&g_decode_status, n < p.N);
        if (p.out_f32) reinterpret_cast<float*>(p.y)[(size_t)tok * p.N + n] = v[i];
        else reinterpret_cast<__nv_bfloat16*>(p.y)[(size_t)tok * p.N + n] = __float2bfloat16_rn(v[i]);
      }
    }
  }

}

template <int MT, bool COMP, bool PERCH, bool XS>
__global__ void __launch_bounds__(kBlockThreads, (MT <= 2 ? 2 : 1)) decode_kernel(const DecodeParams p) {
  extern __shared__ __align__(16) float smem[];
  pdl_launch_dependents();                                 // every block is resident: let the next kernel queue
  if ((int)blockIdx.x < p.Q) {
    // The plain layer keeps the same block split as the compensated one (its
    // producer blocks idle), so forcing the gate to zero reproduces it bit for bit.
    if (COMP && threadIdx.x < kThreads) producer_block<MT>(p, smem);
  } else {
    streamer_block<MT, COMP, PERCH, XS>(p, smem);
  }
}

using KernelFn = void (*)(const DecodeParams);

template <int MT, bool XS>
KernelFn pick_kernel(bool comp, bool perch) {
  if (comp) return perch ? decode_kernel<MT, true, true, XS> : decode_kernel<MT, true, false, XS>;
  return perch ? decode_kernel<MT, false, true, XS> : decode_kernel<MT, false, false, XS>;
}

KernelFn pick(int MT, bool comp, bool perch, bool xs) {
  switch (MT) {
    case 1: return xs ? pick_kernel<1, true>(comp, perch) : pick_kernel<1, false>(comp, perch);
    case 2: return pick_kernel<2, false>(comp, perch);
    default: return pick_kernel<2, false>(comp, perch);
  }
}

// (1-16 tokens: every larger count goes to the tensor-core kernel)
int mt_for(int M) { return M <= 8 ? 1 : 2; }

// Host-side plan: block counts, the tile split and the workspace layout.
struct Plan {
  int device, N, K, G, rank, comp, MT, M;   // key (M matters only for the staged-token variant)
  int xs;                                   // tokens staged in shared memory (M <= 8)
  int Q, P, tiles, nchunks, max_tiles, ng;
  size_t smem;
  size_t off_prod, off_T, off_sync, total;
  KernelFn fn;
  int unsupported;                          // no warp-level plan for this shape (cached)
};

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

size_t xs_smem(int M, int K) {
  return 16 + (size_t)M * (K / 8 + 1) * 16 + 2 * (size_t)M * (K / kChunkK) * 4;
}

size_t streamer_smem(int MT, bool comp, int max_tiles, int ng, int rank, size_t extra = 0) {
  size_t s = extra + (size_t)kWarps * kStages * 2 * 32 * 16; // ring (+ staged tokens)
  s += (size_t)kWarps * MT * 128 * 4;                        // red
  s += (size_t)max_tiles * MT * 128 * 4;                     // ybuf
  if (comp) s += (size_t)MT * 8 * kMaxRank * 4;              // T hi/lo
  s += (size_t)max_tiles * 16 * ng * 2;                      // scales
  s += (size_t)max_tiles * 16 * ((ng + 1) / 2) + 16;         // zero-point bytes (+ alignment)
  if (comp) s += (size_t)max_tiles * 16 * rank * 2 + 16;     // factor-B rows
  return s;
}

int build_plan(const spear_w4_layer& L, int MT, int M, bool comp, bool try_xs, const DeviceInfo& di, Plan* pl) {
  const bool has_rank = L.rank > 0;          // the split depends on this, not on comp_enabled
  pl->MT = MT;
  pl->tiles = L.N / 16;
  pl->nchunks = L.K / kChunkK;
  pl->ng = L.K / L.group_size;
  const bool perch = L.group_size == L.K;
  pl->xs = (MT == 1 && try_xs) ? 1 : 0;
  pl->fn = pick(pl->MT, comp, perch, pl->xs != 0);
  const size_t extra = pl->xs ? xs_smem(M, L.K) : 0;

  // The block count depends on occupancy, which depends on shared memory,
  // which depends on how many tiles one block owns: iterate to a fixed point,
  // then validate occupancy at the final size.
  int blocks = 2 * di.num_sms;
  bool settled = false;
  for (int iter = 0; iter < 8 && !settled; ++iter) {
    if (has_rank) {
      // RT row tiles x S K-slices, enough slices that each producer warp
      // loads its share of A and x in one pass (U 32-k pieces)
      const int RT = (L.rank + 1 + 15) / 16;
      const int U = MT == 1 ? 4 : MT == 2 ? 2 : 1;
      const int S = (4 * pl->nchunks + U * kWarps - 1) / (U * kWarps);
      pl->Q = RT * std::max(1, std::min(S, std::min(kMaxSlices, pl->nchunks)));
    } else {
      pl->Q = 0;
    }
    pl->P = std::max(1, std::min(blocks - pl->Q, pl->tiles));
    pl->max_tiles = (pl->tiles + pl->P - 1) / pl->P;
    if (pl->max_tiles > 64) return fail(SPEAR_ERR_UNSUPPORTED, "decode: too many tiles per block");
    pl->smem = std::max(streamer_smem(pl->MT, has_rank, pl->max_tiles, pl->ng, L.rank, extra),
                        (size_t)kWarps * pl->MT * 128 * 4);
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, pl->fn) != cudaSuccess) return fail(SPEAR_ERR_CUDA, "decode: cudaFuncGetAttributes failed");
    if (pl->smem + fa.sharedSizeBytes > di.smem_optin)
      return fail(SPEAR_ERR_UNSUPPORTED, "decode: shape needs %zu B of shared memory", pl->smem);
    if (int rc = ensure_smem_limit(reinterpret_cast<const void*>(pl->fn), pl->smem)) return rc;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, pl->fn, kBlockThreads, pl->smem) != cudaSuccess ||
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
  pl->off_prod = off; off = align256(off + (size_t)std::max(pl->Q, 1) * Mpad * 16 * 4);
  pl->off_T = off;    off = align256(off + (size_t)Mpad * std::max(L.rank, 1) * 4);
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
        p.comp == comp && p.MT == MT && (MT > 1 || p.M == M)) {
      if (p.unsupported)
        return fail(SPEAR_ERR_UNSUPPORTED, "decode: N=%d K=%d M=%d needs more shared memory than an SM has",
                    L.N, L.K, M);
      *out = p;
      return SPEAR_OK;
    }
  Plan p{};
  // staged tokens when they are small enough to keep two blocks per SM
  // (M <= 8, M K 2 <= 48 KB), else tokens from L1
  const bool try_xs = MT == 1 && xs_smem(M, L.K) <= 48 * 1024;
  int rc = build_plan(L, MT, M, comp != 0, try_xs, di, &p);
  if (rc != SPEAR_OK && MT == 1) rc = build_plan(L, MT, M, comp != 0, false, di, &p);
  p.device = di.device; p.N = L.N; p.K = L.K; p.G = L.group_size; p.rank = L.rank; p.comp = comp; p.M = M;
  p.MT = MT;
  if (rc != SPEAR_OK) {
    if (rc != SPEAR_ERR_UNSUPPORTED) return rc;
    p.unsupported = 1;                     // remembered: later calls take the other kernel at once
    if (cache.size() > 4096) cache.clear();
    cache.push_back(p);
    return rc;
  }
  if (log_plans())
    fprintf(stderr, "[spear] decode plan N=%d K=%d G=%d rank=%d comp=%d M=%d: MT=%d xs=%d Q=%d P=%d max_tiles=%d "
            "smem=%zu\n", L.N, L.K, L.group_size, L.rank, comp, M, p.MT, p.xs, p.Q, p.P, p.max_tiles, p.smem);
  if (cache.size() > 4096) cache.clear();
  cache.push_back(p);
  *out = p;
  return SPEAR_OK;
}

}  // namespace

// Token counts from which the tensor-core kernel (decode_tc.cu) serves the
// call: from there on its MMA throughput beats the warp-level MMAs below,
// whose token fragments are reloaded for every 16 weight rows (measured on
// the Llama-7B shapes: at 24 and 32 tokens the tensor-core kernel takes
// 0.6-0.8x the time, at 16 tokens the warp-level one wins).
#ifndef SPEAR_TC_MIN_M
#define SPEAR_TC_MIN_M 17
#endif
constexpr int kTcMinM = SPEAR_TC_MIN_M;

// The warp-level kernel stages the scales, zero points and factor-B rows of
// all its tiles at once; where that does not fit in shared memory (layers so
// wide that a block owns too many 16-row tiles) the tensor-core kernel, which
// takes any M <= 64, serves the call.
bool use_tc(const spear_w4_layer& L, int M) {
  if (M >= kTcMinM) return true;
  char saved[512];
  snprintf(saved, sizeof(saved), "%s", spear_last_error());
  Plan pl;
  const int rc = get_plan(L, M, &pl);
  if (rc == SPEAR_ERR_UNSUPPORTED) {
    set_last_error(saved);                 // the probe is not this call's failure
    return true;
  }
  return false;
}

int decode_workspace_bytes(const spear_w4_layer& L, int M, size_t* bytes) {
  if (decode_tm_supports(L, M) || decode_ks_supports(L, M)) {   // the cluster K-split kernels need no workspace
    *bytes = 0;
    return SPEAR_OK;
  }
  if (use_tc(L, M)) return decode_tc_workspace_bytes(L, M, bytes);
  Plan pl;
  if (int rc = get_plan(L, M, &pl)) return rc;
  *bytes = pl.total;
  return SPEAR_OK;
}

int launch_decode(const spear_w4_layer& L, const uint16_t* x, int M, void* y, int out_f32, void* ws,
                  size_t ws_bytes, cudaStream_t st, bool overlap) {
  if (decode_tm_supports(L, M)) return launch_decode_tm(L, x, M, y, out_f32, st, overlap);
  if (decode_ks_supports(L, M)) return launch_decode_ks(L, x, M, y, out_f32, st, overlap);
  if (use_tc(L, M)) return launch_decode_tc(L, x, M, y, out_f32, ws, ws_bytes, st, overlap);
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
  p.gh = L.gate_hidden; p.gw1 = L.gate_w1; p.gc1 = L.gate_c1; p.gw2 = L.gate_w2; p.gc2 = L.gate_c2;
  p.Q = pl.Q; p.P = pl.P; p.tiles = pl.tiles; p.nchunks = pl.nchunks;
  p.max_tiles = pl.max_tiles; p.ng = pl.ng;
  char* base = reinterpret_cast<char*>(ws);
  p.ws_sync = reinterpret_cast<unsigned*>(base + pl.off_sync);
  p.ws_prod = reinterpret_cast<float*>(base + pl.off_prod);
  p.ws_T = reinterpret_cast<float*>(base + pl.off_T);
  p.wait_ns = wait_limit_ns(kWaitLimitNs);
  p.smem_bytes = pl.smem;

  if (int rc = ensure_smem_limit(reinterpret_cast<const void*>(pl.fn), pl.smem)) return rc;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(pl.Q + pl.P);
  cfg.blockDim = dim3(kBlockThreads);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 1 : 0;
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
// symbol itself is only a host-side stand-in).  No device work: every call
// clears the synchronisation words on its own stream, and the kernels write
// the rest of the scratch before they read it.
int noalloc_scratch(void** out) {
  int dev = 0;
  if (int rc = cuda_check(cudaGetDevice(&dev), "cudaGetDevice")) return rc;
  if (dev < 0 || dev >= 64) return fail(SPEAR_ERR_UNSUPPORTED, "device index %d", dev);
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* ptr = nullptr;
    if (int rc = cuda_check(cudaGetSymbolAddress((void**)&ptr, g_noalloc_scratch), "decode scratch address"))
      return rc;
    g_noalloc_ptr[dev] = ptr;
  }
  *out = g_noalloc_ptr[dev];
  return SPEAR_OK;
}
}  // namespace

int launch_decode_noalloc(const spear_w4_layer& L, const uint16_t* x, int M, void* y, int out_f32,
                          cudaStream_t st) {
  // the cluster K-split kernel keeps everything it exchanges on chip
  if (decode_tm_supports(L, M)) return launch_decode_tm(L, x, M, y, out_f32, st, false);
  if (decode_ks_supports(L, M)) return launch_decode_ks(L, x, M, y, out_f32, st, false);
  size_t total = 0, sync_bytes = 0;
  if (use_tc(L, M)) {
    if (int rc = decode_tc_workspace_bytes(L, M, &total)) return rc;
    sync_bytes = decode_tc_sync_bytes();
  } else {
    Plan pl;
    if (int rc = get_plan(L, M, &pl)) return rc;
    total = pl.total;
    sync_bytes = pl.off_prod;
  }
  if (total > kNoallocScratchBytes)
    return fail(SPEAR_ERR_UNSUPPORTED,
                "decode_noalloc: N=%d K=%d M=%d needs %zu B of scratch; the built-in scratch holds %zu B",
                L.N, L.K, M, total, kNoallocScratchBytes);
  void* ws = nullptr;
  if (int rc = noalloc_scratch(&ws)) return rc;
  // the synchronisation words must start at zero
  if (int rc = cuda_check(cudaMemsetAsync(ws, 0, sync_bytes, st), "decode scratch clear")) return rc;
  // (after a memset, so no launch overlap)
  return launch_decode(L, x, M, y, out_f32, ws, kNoallocScratchBytes, st, false);
}

int read_and_clear_status_decode(unsigned* out, cudaStream_t st) {
  void* addr = nullptr;
  if (int rc = cuda_check(cudaGetSymbolAddress(&addr, g_decode_status), "decode status address")) return rc;
  if (int rc = cuda_check(cudaMemcpyAsync(out, addr, sizeof(unsigned), cudaMemcpyDeviceToHost, st), "read decode status")) return rc;
  if (int rc = cuda_check(cudaStreamSynchronize(st), "read decode status")) return rc;
  return cuda_check(cudaMemsetAsync(addr, 0, sizeof(unsigned), st), "clear decode status");
}

}  // namespace spear
