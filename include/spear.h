/*
 * spear.h -- C ABI of the GB300 (sm_103a) library for SPEAR's gated 4-bit
 * weight-quantized linear layer with an input-adaptive low-rank error
 * compensator.
 *
 * Source of the method: "SPEAR: A System for Post-Quantization Error-Adaptive
 * Recovery Enabling Efficient Low-Bit LLM Serving" (gist.science explainer of
 * the paper).  Technical Summary 2.1 A gives the compensated effective weight
 * W + alpha * B * diag(gate) * A with a per-token gate; 2.1 B the
 * entropy-aware module selection on CKA damage scores; 2.2 A the phase-aware
 * dispatch (decode: compensator fused into the low-bit GEMM epilogue, one
 * kernel; prefill: compensator as a separate kernel overlapped with the GEMM
 * through a CUDA graph); 2.2 C the SLO-constrained chunk size; 3.1 the RTN
 * per-channel int4 setting.
 *
 * Per token x (one row of x [M][K]) every linear call computes
 *
 *     y = dequant(Wq) x  +  alpha * g(x) * B (A x),   g(x) = sigmoid(w_g . x + b_g)
 *
 * with the scalar gate above by default; a layer with gate_hidden > 0 takes
 * the explainer's vector gate instead, a bottleneck MLP gamma on A x applied
 * per rank component (see spear_w4_layer).
 *
 * Conventions
 *  - Every function returns a spear_status code (0 = SPEAR_OK).  On failure
 *    spear_last_error() gives a one-line, thread-local description.
 *  - Buffers are owned by the caller.  "device" pointers must point into
 *    device memory of the current CUDA device and be 16-byte aligned; "host"
 *    pointers are ordinary host memory.  Nothing here allocates or frees
 *    device memory; calls that need scratch take a caller workspace.
 *  - Device work is queued on the given stream (a cudaStream_t passed as
 *    void*, NULL = legacy default stream) and returns without synchronising.
 *    Kernel-side failures (a bounded wait that ran out, a non-finite weight
 *    seen while packing) are recorded in a device status word that
 *    spear_get_device_status() reads back.
 *  - bf16 and fp16 tensors are passed as uint16_t bit patterns.
 *  - Shapes: K % 128 == 0, N % 64 == 0, group_size == K (per output channel)
 *    or group_size == 128; rank in {0, 16, 32, 64}.
 */
#ifndef SPEAR_H
#define SPEAR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int spear_status;
enum {
  SPEAR_OK = 0,
  SPEAR_ERR_INVALID_ARG = 1,   /* bad shape, NULL or misaligned pointer     */
  SPEAR_ERR_UNSUPPORTED = 2,   /* valid call outside what the kernels cover */
  SPEAR_ERR_WORKSPACE = 3,     /* workspace missing or too small            */
  SPEAR_ERR_CUDA = 4,          /* a CUDA runtime call failed                */
  SPEAR_ERR_TIMEOUT = 5,       /* a bounded device-side wait gave up        */
  SPEAR_ERR_BOUNDS = 6         /* an index check of the debug build failed  */
};

/* Prefill modes (Technical Summary 2.2 A, "semi-fused" prefill). */
enum {
  SPEAR_PREFILL_AUTO = 0,    /* FUSED: the faster mode at every measured shape
                                (Llama-7B projections, M = 512 .. 8192)        */
  SPEAR_PREFILL_FUSED = 1,   /* gate/down-projection pass, then one GEMM whose
                                K loop is extended by the rank-r up-projection */
  SPEAR_PREFILL_STREAM = 2   /* W4 GEMM on `stream` while the compensator's
                                down-projection runs on `stream_aux`; joined by
                                an up-projection-and-add kernel                */
};

/* Output element type of y. */
enum { SPEAR_OUT_BF16 = 0, SPEAR_OUT_F32 = 1 };

/*
 * One quantized linear layer with its compensator (all pointers device).
 *   qweight : uint8 [N][K/2]; byte = u[k even] | u[k odd] << 4, code u in 0..15
 *   scales  : fp16  [N][K/group_size]
 *   zeros   : uint8 [N][ceil(K/group_size/2)], zero points packed like the
 *             codes (low nibble = even group); NULL when symmetric (zero 8)
 *   A       : bf16 [rank][K]   (down-projection)
 *   B       : bf16 [N][rank]   (up-projection)
 *   w_g     : bf16 [K]         (gate weights), b_g gate bias, alpha scale
 *   comp_enabled == 0 or rank == 0 gives the plain W4 layer (A, B, w_g unused).
 */
typedef struct spear_w4_layer {
  int N, K, group_size, symmetric;
  const uint8_t* qweight;
  const uint16_t* scales;
  const uint8_t* zeros;
  int rank;
  const uint16_t* A;
  const uint16_t* B;
  const uint16_t* w_g;
  float b_g, alpha;
  int comp_enabled;
  /* The pages' vector gate (Technical Summary 2.1 A: B diag(gamma(A x)) A,
   * gamma a bottleneck MLP), used when gate_hidden > 0:
   *   t = A x,  gamma(t) = sigmoid(gate_w2 relu(gate_w1 t + gate_c1) + gate_c2),
   *   correction = alpha B (gamma(t) * t)   (elementwise product, per token);
   * device fp32 arrays gate_w1 [gate_hidden][rank], gate_c1 [gate_hidden],
   * gate_w2 [rank][gate_hidden], gate_c2 [rank]; 1 <= gate_hidden <= 32.
   * w_g and b_g are then unused (w_g may be NULL).  gate_hidden = 0 selects
   * the scalar gate g = sigmoid(w_g . x + b_g) and leaves these unread. */
  int gate_hidden;
  const float* gate_w1;
  const float* gate_c1;
  const float* gate_w2;
  const float* gate_c2;
} spear_w4_layer;

/* Byte sizes of the three packed buffers for an N x K weight. */
spear_status spear_pack_w4_sizes(int N, int K, int group_size, int symmetric,
                                 size_t* qweight_bytes, size_t* scales_bytes,
                                 size_t* zeros_bytes);

/*
 * Round-to-nearest int4 quantisation and packing of W (device fp32 [N][K],
 * row-major).  Per group of group_size consecutive k in a row:
 *   symmetric : s = fp16_round_up(max|w| / 7), u = clamp(rint(w/s), -8, 7) + 8
 *   asymmetric: lo = min(min w, 0), hi = max(max w, 0),
 *               s = fp16_round_up((hi - lo) / 15), z = clamp(rint(-lo/s), 0, 15),
 *               u = clamp(rint(w/s) + z, 0, 15)
 * (fp32 IEEE division, rint = round half to even; an all-zero group stores
 * s = 0 and the zero point as its codes).  Writes qweight, scales and, when
 * asymmetric, zeros (device).  A non-finite weight or a scale beyond the fp16
 * range is reported through spear_get_device_status (SPEAR_ERR_INVALID_ARG).
 */
spear_status spear_pack_w4(const float* W, int N, int K, int group_size, int symmetric,
                           uint8_t* qweight, uint16_t* scales, uint8_t* zeros,
                           void* stream);

/*
 * Decode (Technical Summary 2.2 A, decode phase, M small): ONE kernel launch
 * streams the int4 weights, computes g(x) and A x for every token in the same
 * launch and adds alpha*g*B(Ax) in the epilogue.  0 <= M <= 64 (M = 0: no work, SPEAR_OK).
 *   x : device bf16 [M][K];  y : device [M][N], bf16 or fp32 (out_dtype).
 * M <= 16 runs on warp-level MMAs; M >= 17 on the tcgen05 tensor cores.
 * The thread blocks of the launch exchange the M x (rank+1) down-projection
 * and the gated term T derived from it through `workspace` (device, at least
 * spear_decode_workspace_bytes()).
 * The workspace must be zeroed once before its first use
 * (spear_workspace_init) and is left ready for the next call; two calls that
 * run at the same time must not share one.  After a SPEAR_ERR_TIMEOUT device
 * status, zero it again.
 * Every block of a launch stays resident at once; a shape too wide for that
 * (e.g. N = 131072 at 12 tokens) returns SPEAR_ERR_UNSUPPORTED.
 * Some launches carry the activations in fp16 (M <= 8 with M*K*2 <= 48 KB,
 * and M >= 17); any finite bf16 input is still computed.  With M <= 8 a
 * token whose max |x| reaches 2^15 enters as x 2^-e (a power of two, exact in
 * fp16 for every value above 2^-24 2^e) and its outputs are multiplied by
 * 2^e.  With M >= 17 a token holding a value of 65504 or more (beyond fp16)
 * has its main-term partial sums recomputed in fp32 from the int4 codes and
 * the bf16 values, outside the tensor cores (slower, for such tokens only).
 * A non-finite token value is reported as SPEAR_ERR_INVALID_ARG through
 * spear_get_device_status.
 */
spear_status spear_decode_workspace_bytes(const spear_w4_layer* L, int M, size_t* bytes);
spear_status spear_linear_decode(const spear_w4_layer* L, const uint16_t* x, int M,
                                 void* y, int out_dtype, void* workspace, size_t ws_bytes,
                                 void* stream);

/*
 * Decode for callers that cannot allocate device memory.  (The paper has no
 * counterpart: this is a deployment convenience of this library.)
 * Some callers cannot allocate when they call the layer -- a plugin hosted
 * by a framework that owns the device allocator, a runtime that plans every
 * buffer before serving and forbids allocation afterwards, code on a
 * latency-critical path where an allocation could synchronise the device.
 * This call computes exactly what spear_linear_decode computes, but keeps its
 * scratch in one fixed 8 MiB array inside the library (every GPU that loads
 * the library holds it until the process exits) instead of a workspace.
 *   - A shape whose decode scratch exceeds 8 MiB is rejected with
 *     SPEAR_ERR_UNSUPPORTED; spear_last_error() gives the bytes needed.
 *   - The first call on a device sets the scratch up: it looks up the
 *     array's device address (host work only, no device work); make that
 *     first call before any stream capture.
 *   - Every call clears the scratch's synchronisation words on `stream` and
 *     otherwise reuses what the previous call left there.  All calls share
 *     the one array: calls that overlap on the GPU (other streams, other host
 *     threads) race and give wrong results.
 *   - After spear_get_device_status reports SPEAR_ERR_TIMEOUT, synchronise
 *     the device before the next call here: a thread block of the launch
 *     that timed out may still write the shared array.
 *   - This call never uses launch overlap (spear_set_launch_overlap): the
 *     clear on `stream` must finish before the kernel starts.
 * Nothing here allocates device memory.
 */
spear_status spear_linear_decode_noalloc(const spear_w4_layer* L, const uint16_t* x, int M,
                                         void* y, int out_dtype, void* stream);

/*
 * Prefill (Technical Summary 2.2 A, prefill phase, M large): tcgen05 tensor-core
 * GEMM over int4 tiles dequantized in shared memory, plus the compensator in
 * one of the modes above.  M >= 0 (M = 0: no work, SPEAR_OK).
 *   x : device bf16 [M][K];  y : device [M][N], bf16 or fp32.
 *   The main GEMM runs on fp16 operands with fp32 accumulation: each token is
 *   copied to fp16 as x 2^-e, the smallest power-of-two scale that brings its
 *   max |x| below 2^15 (exact for every value above 2^-24 2^e; e = 0 for most
 *   tokens), and its outputs are multiplied by 2^e; a group-scaled weight is
 *   rounded once to fp16.  A non-finite token value is reported as
 *   SPEAR_ERR_INVALID_ARG through spear_get_device_status.  The compensator
 *   terms stay in bf16 with fp32 accumulation.
 *   workspace : device, at least spear_prefill_workspace_bytes(); no zeroing
 *               needed.  stream_aux is used by SPEAR_PREFILL_STREAM only (it
 *               may be NULL otherwise); the call orders it after `stream` and
 *               joins it back, so the call behaves as one operation on `stream`.
 */
spear_status spear_prefill_workspace_bytes(const spear_w4_layer* L, int M, int mode,
                                           size_t* bytes);
spear_status spear_linear_prefill(const spear_w4_layer* L, const uint16_t* x, int M,
                                  void* y, int out_dtype, int mode,
                                  void* workspace, size_t ws_bytes,
                                  void* stream, void* stream_aux);

/* Zero a decode workspace (device) on `stream`. */
spear_status spear_workspace_init(void* workspace, size_t bytes, void* stream);

/*
 * Launch overlap for chains of decode calls (process-wide, default off).
 * With enable != 0, spear_linear_decode launches use programmatic dependent
 * launch (spear_linear_decode_noalloc never does): a decode kernel may start while the kernel
 * before it on the same stream is still finishing, and streams its weights
 * meanwhile; it waits for that kernel to complete (with its memory visible)
 * before it reads x, touches the workspace or writes y.  The caller
 * guarantees that the kernel immediately before a decode call on the stream
 * does not write that layer's qweight, scales, zeros, A, B or w_g.
 * Host only; takes effect for launches issued afterwards (also inside stream
 * capture, where it becomes a programmatic graph edge).
 */
spear_status spear_set_launch_overlap(int enable);

/*
 * Limit of the device-side waits on other thread blocks (process-wide).  A
 * decode launch's blocks wait for the down-projection that other blocks of
 * the same launch publish (and the cluster kernels for their peers); each
 * such wait gives up after `ns` nanoseconds, records SPEAR_ERR_TIMEOUT in the
 * device status word and lets its kernel finish with the compensator term
 * left out.  ns = 0 restores the defaults (200 ms; 2 s in the cluster
 * kernels).  For tests and diagnostics: a limit shorter than a legitimate
 * wait makes correct calls fail.  Host only; takes effect for launches issued
 * afterwards.
 */
spear_status spear_set_wait_limit_ns(uint64_t ns);

/*
 * Module selection (Technical Summary 2.1 B), host only.  damage[L] >= 0 is a
 * per-module quantisation-damage score, cost[L] > 0 the bytes one unit of
 * rank costs in module i.  The damage distribution p_i = d_i / sum d sets
 * k = clamp(round(exp(entropy(p))), 1, L) modules; they are the k best by
 * p_i / (cost_i / mean cost) (ties: lower index), and all get the largest
 * rank that is a multiple of 16 in [rank_min, rank_max] with
 * rank * sum(selected cost) <= budget_bytes; if even the smallest rank does
 * not fit, the worst selected module is dropped and the rank chosen again.
 * Writes mask_out[L] (1 = carries a compensator) and rank_out[L] (0 when
 * unselected), both host.
 */
spear_status spear_layer_select_mask(const float* damage, const float* cost, int L,
                                     double budget_bytes, int rank_min, int rank_max,
                                     uint8_t* mask_out, int* rank_out);

/*
 * Linear centred kernel alignment (Technical Summary 2.1 B: CKA is the
 * training-free proxy for the quality a module loses to quantisation), host
 * only.  X [n][dx] and Y [n][dy] are fp32, one row per token; with Xc, Yc
 * their column-centred forms
 *   *cka_out = ||Xc^T Yc||_F^2 / (||Xc^T Xc||_F ||Yc^T Yc||_F)   (in [0, 1]),
 * computed in fp64.  A module's damage score for spear_layer_select_mask is
 * 1 - CKA(its reference output, its quantised output) on the same tokens.
 * n >= 2; non-finite inputs or an input without variance are rejected.
 */
spear_status spear_linear_cka(const float* X, const float* Y, int n, int dx, int dy, double* cka_out);

/*
 * A module's damage score for spear_layer_select_mask (Technical Summary
 * 2.1 B), host only: *damage_out = 1 - CKA(X_ref, Y_quant) with the same
 * arguments, checks and arithmetic as spear_linear_cka (X_ref: the module's
 * reference output, Y_quant: its quantised output on the same n tokens).
 */
spear_status spear_cka_damage(const float* X_ref, const float* Y_quant, int n, int dx, int dy,
                              double* damage_out);

/*
 * SLO-constrained chunk selection (Technical Summary 2.2 C), host only.
 * A latency curve holds n >= 1 measured points (M[i], us[i]) of one layer
 * (M strictly increasing, us >= 0); between points the latency is linear in
 * M, outside them it continues the line through the two nearest points (one
 * point: constant).  For a step with D = decode_tokens decode tokens and a
 * prefill chunk of C tokens the predicted step latency is
 *   C > 0:  sum over layers of prefill[l](C + D)   (one mixed pass, prefill path)
 *   C = 0:  sum over layers of decode[l](D)        (decode path; 0 if D = 0)
 * chunk_out receives the largest C in choices[nchoices] (C >= 0) whose step
 * latency is <= itl_target_us; if none is, the smallest C.  step_us_out (may
 * be NULL) receives that C's predicted latency.  A layer's curves reflect its
 * compensator (or its absence), so the choice follows the EC density.
 */
typedef struct spear_latency_curve {
  int n;
  const int* M;
  const float* us;
} spear_latency_curve;

spear_status spear_chunk_select(const spear_latency_curve* prefill, const spear_latency_curve* decode,
                                int nlayers, int decode_tokens, const int* choices, int nchoices,
                                double itl_target_us, int* chunk_out, double* step_us_out);

/*
 * Reads and clears the device status word of the current device
 * (synchronises `stream`).  *out = SPEAR_OK, or the first kernel-side error
 * recorded since the last read.
 */
spear_status spear_get_device_status(int* out, void* stream);

/* Static, human-readable name of a status code. */
const char* spear_status_string(int status);

/* Thread-local description of the last failing call on this thread. */
const char* spear_last_error(void);

/* Library version as "major.minor.patch". */
const char* spear_version(void);

#ifdef __cplusplus
}
#endif
#endif /* SPEAR_H */
