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
};

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

// Four bf16x2 values holding (128 + nibble) for the 8 nibbles of `w`:
// out[i] = (128 + nib_i, 128 + nib_{i+4}) for i = 0..3 (nib_j = bits 4j..4j+3).
__device__ __forceinline__ void nibbles_to_bf16x2_biased(uint32_t w, uint32_t (&out)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) out[i] = ((w >> (4 * i)) & 0x000F000Fu) | 0x43004300u;
}

// The vector gate (Technical Summary 2.1 A: gamma is a bottleneck MLP on the
// rank-r code t = A x), for ntok tokens at once, in two phases with a barrier
// of the calling threads [tid0, tid0 + nthreads) between and after them:
//   vector_gate_hidden:  hid[m][i] = relu(c1[i] + sum_j W1s[i][j] t[m][j])   [ntok][h]
//   vector_gate_apply:   t[m][j] *= sigmoid(c2[j] + sum_i W2s[j][i] hid[m][i])
// t[m][j] sits at t[m * tm + j * tj] (shared memory); W1s [h][r] and W2s
// [r][h] are staged in shared memory (stage_gate_weights); c1 [h], c2 [r] are
// fp32 in global memory.  fp32 accumulation in index order; every (token,
// unit) pair belongs to one thread, so apply may overwrite t in place.
__device__ __forceinline__ void vector_gate_hidden(const float* t, int tm, int tj, int ntok, int r, int h,
                                                   const float* W1s, const float* c1, float* hid, int tid,
                                                   int nthreads) {
  for (int e = tid; e < ntok * h; e += nthreads) {
    const int m = e / h, i = e % h;
    float acc = __ldg(c1 + i);
    for (int j = 0; j < r; ++j) acc = fmaf(W1s[i * r + j], t[m * tm + j * tj], acc);
    hid[e] = fmaxf(acc, 0.0f);
  }
}
__device__ __forceinline__ void vector_gate_apply(float* t, int tm, int tj, int ntok, int r, int h,
                                                  const float* W2s, const float* c2, const float* hid, int tid,
                                                  int nthreads) {
  for (int e = tid; e < ntok * r; e += nthreads) {
    const int m = e / r, j = e % r;
    float acc = __ldg(c2 + j);
    for (int i = 0; i < h; ++i) acc = fmaf(W2s[j * h + i], hid[m * h + i], acc);
    t[m * tm + j * tj] *= 1.0f / (1.0f + expf(-acc));
  }
}

// Copies the gate's W1 [h][r] and W2 [r][h] (fp32, global) into shared memory
// with threads [tid0, tid0 + nthreads) of the block, eight loads in flight per
// thread; the caller synchronises those threads afterwards.
__device__ __forceinline__ void stage_gate_weights(const float* W1, const float* W2, int r, int h, float* W1s,
                                                   float* W2s, int tid, int nthreads) {
  const int n = h * r;
  for (int e0 = 0; e0 < 2 * n; e0 += 8 * nthreads) {
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = e0 + tid + i * nthreads;
      v[i] = e < n ? __ldg(W1 + e) : e < 2 * n ? __ldg(W2 + (e - n)) : 0.0f;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = e0 + tid + i * nthreads;
      if (e < n) W1s[e] = v[i];
      else if (e < 2 * n) W2s[e - n] = v[i];
    }
  }
}

}  // namespace spear
