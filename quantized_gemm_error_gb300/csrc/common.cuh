// common.cuh -- small device helpers shared by the library's kernels
// (sm_103a).  Nothing here is shared with the CPU oracle.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace spear {

// Device-side status codes (same numbering as the C ABI's spear_status).
enum : unsigned {
  DEV_OK = 0,
  DEV_ERR_INVALID = 1,
  DEV_ERR_TIMEOUT = 5,
  DEV_ERR_BOUNDS = 6,
};

// Index checks of the debug build (compiled with -DSPEAR_DEBUG_CHECKS): a
// check that fails records SPEAR_ERR_BOUNDS in the kernel's status word and
// the kernel carries on (no trap).  The release build evaluates nothing.
#ifdef SPEAR_DEBUG_CHECKS
#define SPEAR_CHECK(word, cond)                                              \
  do {                                                                       \
    if (!(cond)) ::spear::record_status((word), ::spear::DEV_ERR_BOUNDS);   \
  } while (0)
#else
#define SPEAR_CHECK(word, cond) \
  do {                          \
  } while (0)
#endif

// A pointer into shared memory moved up to the next multiple of `align`
// bytes (a power of two) by offsetting the original pointer.  (Rounding an
// integer copy of the pointer instead would hide its address space from the
// compiler, and every access through the result would become a slower
// generic load or store.)
template <typename T>
__device__ __forceinline__ T* smem_align_up(T* p, uint32_t align) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
  return reinterpret_cast<T*>(reinterpret_cast<uint8_t*>(p) + ((align - (a & (align - 1))) & (align - 1)));
}

// Keeps the first error: later errors do not overwrite it.
__device__ __forceinline__ void record_status(unsigned* word, unsigned code) {
  atomicCAS(word, 0u, code);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_gpu(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Atomic add with acquire-release semantics at GPU scope (returns the old value).
__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// 16-byte load through L1 (read-only path): for small operands reused by
// many warps (activations, low-rank factors).
__device__ __forceinline__ uint4 ldg16(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// 16-byte asynchronous global->shared copy that bypasses L1 (streamed data).
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
// 4-byte asynchronous global->shared copy through L1 (small operands).
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
  unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(s), "l"(gmem) : "memory");
}
// Programmatic dependent launch: let the next kernel on the stream start
// launching / wait until the previous kernel completed with its memory
// visible.  Both are no-ops for a launch without the programmatic attribute.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Prefetch of the 128-byte line holding `ptr` into L1 (no register, no wait).
__device__ __forceinline__ void prefetch_l1(const void* ptr) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(reinterpret_cast<uint64_t>(ptr)));
}

// Bulk prefetch of [ptr, ptr + bytes) into L2 (16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void prefetch_l2(const void* ptr, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(ptr)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// D(16x8, f32) += A(16x16, bf16, row) * B(16x8, bf16, col).
// Lane (g = lane/4, c = lane%4) holds a0 = A[g][2c..2c+1], a1 = A[g+8][2c..],
// a2 = A[g][2c+8..], a3 = A[g+8][2c+8..]; b0 = B[2c..2c+1][g], b1 = B[2c+8..][g];
// d0,d1 = D[g][2c..2c+1], d2,d3 = D[g+8][2c..2c+1].
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Same shape with fp16 A and B (fp32 accumulate).
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// bf16x2 subtraction (exact for the small integers used by the dequantiser).
__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
  __nv_bfloat162 r = __hsub2(*reinterpret_cast<__nv_bfloat162*>(&a), *reinterpret_cast<__nv_bfloat162*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

// Two floats -> bf16x2 (round to nearest even); `lo` lands in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&r);
}

// The two bf16 halves of a bf16x2 word as floats (exact).
__device__ __forceinline__ float bf16x2_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16x2_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// bf16 value of (128 + v) for an integer 0 <= v < 128 in both halves: the
// exponent of 128 with v in the mantissa.  Used as the bias that turns a
// nibble into an exact small integer.
__host__ __device__ constexpr uint32_t bf16x2_bias(uint32_t v) { return (0x4300u | v) * 0x00010001u; }

// Four fp16x2 values holding (1024 + nibble) for the 8 nibbles of `w`:
// out[i] = (1024 + nib_i, 1024 + nib_{i+4}) (fp16 1024 has a mantissa unit of 1).
__device__ __forceinline__ void nibbles_to_f16x2_biased(uint32_t w, uint32_t (&out)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) out[i] = ((w >> (4 * i)) & 0x000F000Fu) | 0x64006400u;
}
__host__ __device__ constexpr uint32_t f16x2_bias(uint32_t v) { return (0x6400u | v) * 0x00010001u; }

__device__ __forceinline__ uint32_t f16x2_sub(uint32_t a, uint32_t b) {
  __half2 r = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t f16x2_mul(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

// Power-of-two token scaling for the fp16 operand copies of the activations:
// a token x_m enters as x_m 2^-e_m with the smallest e_m >= 0 that brings
// max|x_m| below 2^15, which is exact in fp16 for every value above 2^-24 2^e_m
// (bf16 carries 8 significant bits, fp16 11); the fp32 accumulator is
// multiplied by 2^e_m afterwards.  e = 0 for max|x| < 2^15 and for a
// non-finite max (reported separately).
__device__ __forceinline__ int token_scale_exp(float amax) {
  if (!(amax >= 32768.0f) || !(amax <= 3.4e38f)) return 0;
  return (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127 - 14;   // floor(log2 amax) - 14
}
// 2^k as a float, -126 <= k <= 127 (exact)
__device__ __forceinline__ float exp2_int(int k) { return __uint_as_float((uint32_t)(k + 127) << 23); }
// max |x| of 8 bf16 values (NaN propagates as a value above every finite one)
__device__ __forceinline__ float bf16x8_absmax(uint4 v) {
  const uint32_t m = 0x7fff7fffu;
  const uint32_t a = __vmaxu2(__vmaxu2(v.x & m, v.y & m), __vmaxu2(v.z & m, v.w & m));   // bf16 bits order like |x|
  const uint32_t b = __vmaxu2(a, a >> 16);
  return __uint_as_float((b & 0xffffu) << 16);
}

// Four bf16x2 values holding (128 + nibble) for the 8 nibbles of `w`:
// out[i] = (128 + nib_i, 128 + nib_{i+4}) for i = 0..3 (nib_j = bits 4j..4j+3).
__device__ __forceinline__ void nibbles_to_bf16x2_biased(uint32_t w, uint32_t (&out)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) out[i] = ((w >> (4 * i)) & 0x000F000Fu) | 0x43004300u;
}

// The vector gate (Technical Summary 2.1 A: gamma is a bottleneck MLP on the
// rank-r code t = A x), for ntok tokens at once, in two phases with a barrier
// of the calling threads between and after them:
//   hidden:  hid[m][i] = relu(c1[i] + sum_j W1[i][j] t[m][j])
//   apply:   t[m][j] *= sigmoid(c2[j] + sum_i W2[j][i] hid[m][i])
// The fp32 weights are read from the shared-memory copy that
// stage_gate_weights_async makes, laid out so that the loads of a warp hit
// distinct banks (W1 [h][r] and W2 [r][h] as given put a warp's rows a
// multiple of 32 floats apart: 8-way conflicts that made these loops cost
// more than the rest of the tensor-core decode's epilogue):
//   G = [ W1 [h][r + 4] (rows padded) | W2^T [h][r] | c2 [r] | c1 [h] ],
// every part 16-byte aligned when G is (the rank is a multiple of 16).  The
// hidden units sit at hid[m * gate_hid_stride(h) + i].  Every (token, unit)
// element belongs to one thread, so apply may overwrite t in place.
__host__ __device__ constexpr int gate_smem_floats(int r, int h) { return h * (r + 4) + h * r + r + h; }
__host__ __device__ constexpr int gate_hid_stride(int h) { return h | 1; }

struct GateSmem {
  const float *W1, *W2t, *c2, *c1;
  int r, h;
  __device__ GateSmem(const float* G, int r_, int h_)
      : W1(G), W2t(G + h_ * (r_ + 4)), c2(G + h_ * (r_ + 4) + h_ * r_), c1(G + h_ * (r_ + 4) + h_ * r_ + r_),
        r(r_), h(h_) {}
};

// Starts the copy of the gate's W1 [h][r], W2 [r][h], c1 [h], c2 [r] (fp32,
// global) into the layout above as one cp.async group of threads [tid0, tid0
// + nthreads): issued where the kernel starts, so the copy overlaps its main
// work.  Before reading G the caller waits for the group (cp_async_wait<0>)
// and then synchronises those threads.
__device__ __forceinline__ void stage_gate_weights_async(const float* W1, const float* W2, const float* c1,
                                                         const float* c2, int r, int h, float* G, int tid,
                                                         int nthreads) {
  const int n1 = h * (r + 4), n2 = n1 + h * r, n3 = n2 + r, total = gate_smem_floats(r, h);
  for (int e = tid; e < total; e += nthreads) {
    const float* src = nullptr;
    if (e < n1) {
      const int i = e / (r + 4), j = e % (r + 4);
      if (j < r) src = W1 + i * r + j;
    } else if (e < n2) {
      const int i = (e - n1) / r, j = (e - n1) % r;
      src = W2 + j * h + i;
    } else if (e < n3) {
      src = c2 + (e - n2);
    } else {
      src = c1 + (e - n3);
    }
    if (src) cp_async4(G + e, src);
  }
  cp_async_commit();
}

// Token rows t[m][0 .. r) at t + m r (16-byte aligned): 16-byte loads, one
// hidden unit of one token per thread, then four consecutive components of
// one token per thread.  Each dot product is four fp32 partial sums (terms
// q mod 4) added at the end.
__device__ __forceinline__ void vector_gate_hidden_rows(const float* t, int ntok, const GateSmem& g, float* hid,
                                                        int tid, int nthreads) {
  const int r4 = g.r / 4, hs = gate_hid_stride(g.h);
  for (int e = tid; e < ntok * g.h; e += nthreads) {
    const int m = e / g.h, i = e % g.h;
    const float4* w = reinterpret_cast<const float4*>(g.W1 + i * (g.r + 4));
    const float4* tt = reinterpret_cast<const float4*>(t + m * g.r);
    float4 a = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll 4
    for (int q = 0; q < r4; ++q) {
      const float4 wv = w[q], tv = tt[q];
      a.x = fmaf(wv.x, tv.x, a.x);
      a.y = fmaf(wv.y, tv.y, a.y);
      a.z = fmaf(wv.z, tv.z, a.z);
      a.w = fmaf(wv.w, tv.w, a.w);
    }
    hid[m * hs + i] = fmaxf(g.c1[i] + ((a.x + a.y) + (a.z + a.w)), 0.0f);
  }
}
__device__ __forceinline__ void vector_gate_apply_rows(float* t, int ntok, const GateSmem& g, const float* hid,
                                                       int tid, int nthreads) {
  const int r4 = g.r / 4, hs = gate_hid_stride(g.h);
  for (int e = tid; e < ntok * r4; e += nthreads) {
    const int m = e / r4, q = e % r4;
    float4 a = reinterpret_cast<const float4*>(g.c2)[q];
    const float* hh = hid + m * hs;
#pragma unroll 4
    for (int i = 0; i < g.h; ++i) {
      const float4 wv = reinterpret_cast<const float4*>(g.W2t + i * g.r)[q];
      const float hv = hh[i];
      a.x = fmaf(wv.x, hv, a.x);
      a.y = fmaf(wv.y, hv, a.y);
      a.z = fmaf(wv.z, hv, a.z);
      a.w = fmaf(wv.w, hv, a.w);
    }
    float4* tp = reinterpret_cast<float4*>(t + m * g.r) + q;
    float4 tv = *tp;
    tv.x *= 1.0f / (1.0f + expf(-a.x));
    tv.y *= 1.0f / (1.0f + expf(-a.y));
    tv.z *= 1.0f / (1.0f + expf(-a.z));
    tv.w *= 1.0f / (1.0f + expf(-a.w));
    *tp = tv;
  }
}

// Any layout: t[m][j] at t[m * tm + j * tj]; one (token, unit) pair per
// thread, dot products as four partial sums (terms q mod 4).
__device__ __forceinline__ void vector_gate_hidden(const float* t, int tm, int tj, int ntok, const GateSmem& g,
                                                   float* hid, int tid, int nthreads) {
  const int hs = gate_hid_stride(g.h);
  for (int e = tid; e < ntok * g.h; e += nthreads) {
    const int m = e / g.h, i = e % g.h;
    const float* w = g.W1 + i * (g.r + 4);
    const float* tt = t + m * tm;
    float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
#pragma unroll 4
    for (int j = 0; j < g.r; j += 4) {
      a0 = fmaf(w[j], tt[j * tj], a0);
      a1 = fmaf(w[j + 1], tt[(j + 1) * tj], a1);
      a2 = fmaf(w[j + 2], tt[(j + 2) * tj], a2);
      a3 = fmaf(w[j + 3], tt[(j + 3) * tj], a3);
    }
    hid[m * hs + i] = fmaxf(g.c1[i] + ((a0 + a1) + (a2 + a3)), 0.0f);
  }
}
__device__ __forceinline__ void vector_gate_apply(float* t, int tm, int tj, int ntok, const GateSmem& g,
                                                  const float* hid, int tid, int nthreads) {
  const int hs = gate_hid_stride(g.h);
  for (int e = tid; e < ntok * g.r; e += nthreads) {
    const int m = e / g.r, j = e % g.r;
    const float* hh = hid + m * hs;
    float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
    int i = 0;
#pragma unroll 2
    for (; i + 4 <= g.h; i += 4) {
      a0 = fmaf(g.W2t[i * g.r + j], hh[i], a0);
      a1 = fmaf(g.W2t[(i + 1) * g.r + j], hh[i + 1], a1);
      a2 = fmaf(g.W2t[(i + 2) * g.r + j], hh[i + 2], a2);
      a3 = fmaf(g.W2t[(i + 3) * g.r + j], hh[i + 3], a3);
    }
    if (i < g.h) a0 = fmaf(g.W2t[i * g.r + j], hh[i], a0);
    if (i + 1 < g.h) a1 = fmaf(g.W2t[(i + 1) * g.r + j], hh[i + 1], a1);
    if (i + 2 < g.h) a2 = fmaf(g.W2t[(i + 2) * g.r + j], hh[i + 2], a2);
    const float acc = g.c2[j] + ((a0 + a1) + (a2 + a3));
    t[m * tm + j * tj] *= 1.0f / (1.0f + expf(-acc));
  }
}

}  // namespace spear
