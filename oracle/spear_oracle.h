/*
 * spear_oracle.h -- plain CPU reference for the gated W4 + low-rank
 * error-compensated linear layer described in "SPEAR: A System for
 * Post-Quantization Error-Adaptive Recovery Enabling Efficient Low-Bit LLM
 * Serving" (gist.science explainer, Technical Summary section 2.1 A,
 * "Input-Adaptive Error Compensators", effective weight W + alpha*B*diag(gate)*A).
 *
 * TEST INFRASTRUCTURE ONLY.  This library is the parity oracle for the CUDA
 * path.  It shares no code, header, table or helper with the CUDA library and
 * must never be linked into it.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load it.
 *
 * Everything here is deliberately slow and literal: one loop per sum, no
 * blocking, no vectorisation, no reordering.  Accumulation is in double
 * unless a function says otherwise.
 *
 * Encodings (plain C types so the header needs no CUDA):
 *   fp16 values  : uint16_t holding IEEE binary16 bits
 *   bf16 values  : uint16_t holding bfloat16 bits (upper half of a float)
 *   qweight      : uint8_t [N][K/2], byte = u[k even] | (u[k odd] << 4)
 *   scales       : fp16   [N][K/G]
 *   zeros        : uint8_t [N][ceil((K/G)/2)], same nibble order over groups;
 *                  NULL for the symmetric format (zero point 8 implied)
 *
 * Return values: 0 on success, 1 on an invalid argument (bad shape, NULL
 * pointer, non-finite weight, scale overflow).
 */
#ifndef SPEAR_ORACLE_H
#define SPEAR_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Number formats used by the method (exported so the pins can test them). */
uint16_t oracle_f32_to_f16_ru(float f);   /* IEEE binary16, round toward +inf */
float    oracle_f16_to_f32(uint16_t h);
uint16_t oracle_f32_to_bf16_rn(float f);  /* bfloat16, round to nearest even  */
float    oracle_bf16_to_f32(uint16_t b);

/* Round-to-nearest int4 quantisation of one weight matrix W [N][K] (fp32),
 * per group of G consecutive k in a row (G == K: per output channel).
 * sym = 1: scale = fp16_ru(amax/7), code u = clamp(rint(w/s), -8, 7) + 8.
 * sym = 0: lo = min(min w, 0), hi = max(max w, 0), s = fp16_ru((hi-lo)/15),
 *          z = clamp(rint(-lo/s), 0, 15), u = clamp(rint(w/s) + z, 0, 15). */
int oracle_quantize_pack(const float* W, int N, int K, int G, int sym,
                         uint8_t* qweight, uint16_t* scales, uint8_t* zeros);

/* Codes u[N][K] (0..15) read back from the packed bytes. */
int oracle_unpack_codes(const uint8_t* qweight, int N, int K, uint8_t* codes);

/* Zero points z[N][K/G] (8 for the symmetric format). */
int oracle_unpack_zeros(const uint8_t* zeros, int N, int K, int G, int sym, uint8_t* z);

/* Dequantised weights dq[n][k] = (u - z) * s, exact in double. */
int oracle_dequant(const uint8_t* qweight, const uint16_t* scales, const uint8_t* zeros,
                   int N, int K, int G, int sym, double* dq);

/* The layer, per token m (x [M][K] bf16):
 *   s_m    = w_g . x_m + b_g
 *   g_m    = 1 / (1 + exp(-s_m))
 *   t_m    = A x_m                      (A [r][K] bf16)
 *   y[m,n] = sum_k dq[n][k] x[m][k]  +  alpha * g_m * sum_j B[n][j] t_m[j]
 * comp_enabled == 0 or r == 0 drops the second term.
 * n_idx (may be NULL = all N rows, n_count ignored) selects the output
 * columns; y and corr are [M][n_count].  corr (may be NULL) receives the
 * second term alone, gate (may be NULL) receives g_m [M].
 * accum_double = 1: every sum in double.  accum_double = 0: the main sum and
 * t_m, s_m are accumulated in float, ascending k (no fused multiply-add).
 * nthreads <= 1 runs on the calling thread; otherwise rows are split evenly. */
int oracle_linear(int N, int K, int G, int sym,
                  const uint8_t* qweight, const uint16_t* scales, const uint8_t* zeros,
                  int r, const uint16_t* A, const uint16_t* B, const uint16_t* w_g,
                  float b_g, float alpha, int comp_enabled,
                  const uint16_t* x, int M,
                  const int* n_idx, int n_count,
                  int accum_double, int nthreads,
                  double* y, double* corr, double* gate);

/* The paper's own gate form (Technical Summary 2.1 A): a bottleneck MLP on
 * the rank-r code, gamma(Ax) = sigmoid(W2 relu(W1 (Ax) + c1) + c2), applied
 * per rank component:  y = dq x + alpha * B diag(gamma(Ax)) A x.
 * W1 [h][r], c1 [h], W2 [r][h], c2 [r] are fp32. */
int oracle_linear_vector_gate(int N, int K, int G, int sym,
                              const uint8_t* qweight, const uint16_t* scales, const uint8_t* zeros,
                              int r, const uint16_t* A, const uint16_t* B,
                              int h, const float* W1, const float* c1,
                              const float* W2, const float* c2, float alpha,
                              const uint16_t* x, int M, int nthreads,
                              double* y, double* gamma_out);

/* Entropy-aware module selection (Technical Summary 2.1 B):
 *   p_i = d_i / sum d,  H = -sum p_i ln p_i,  k = clamp(round(exp H), 1, L)
 *   score_i = p_i / (c_i / mean c); take the k best scores (ties: lower i);
 *   rank r = largest multiple of 16 in [rank_min, rank_max] with
 *   r * sum_{selected} c_i <= budget; if none fits, drop the worst selected
 *   module and retry.  Unselected modules get mask 0, rank 0. */
int oracle_layer_select_mask(const float* damage, const float* cost, int L,
                             double budget_bytes, int rank_min, int rank_max,
                             uint8_t* mask_out, int* rank_out);

#ifdef __cplusplus
}
#endif
#endif
