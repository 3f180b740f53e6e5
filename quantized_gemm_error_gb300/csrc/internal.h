// internal.h -- host-side interface between the C ABI (api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "spear.h"

namespace spear {

// Records a thread-local error message and returns `status`.
int fail(int status, const char* fmt, ...);
// Puts back a thread-local error message saved earlier (after an internal
// probe that failed on purpose).
void set_last_error(const char* msg);
// Maps a CUDA error to SPEAR_ERR_CUDA with a message (SPEAR_OK if e == cudaSuccess).
int cuda_check(cudaError_t e, const char* what);

// Device properties of the current device, cached per device.
struct DeviceInfo {
  int device;
  int num_sms;
  int cc_major, cc_minor;
  size_t smem_optin;
};
int device_info(DeviceInfo* out);

// True when the environment variable SPEAR_LOG_PLANS is set to a non-empty
// value other than "0": launch plans are then printed to stderr once each.
bool log_plans();

// Programmatic dependent launch for decode kernels (spear_set_launch_overlap).
void set_launch_overlap(bool on);
bool launch_overlap();
// Limit of the waits on other thread blocks (spear_set_wait_limit_ns): the
// set value, or `default_ns` while none is set.
uint64_t wait_limit_ns(uint64_t default_ns);

// Raises (never lowers) the dynamic shared-memory limit of kernel `fn` on the
// current device to at least `bytes`.  Launches captured in CUDA graphs keep
// the size they were captured with, so a limit that a later plan lowered
// would make an earlier graph fail; the limit therefore only grows.
int ensure_smem_limit(const void* fn, size_t bytes);

// ---- pack.cu
int launch_pack_w4(const float* W, int N, int K, int G, int sym, uint8_t* qweight,
                   uint16_t* scales, uint8_t* zeros, cudaStream_t st);
int read_and_clear_status_pack(unsigned* out, cudaStream_t st);

// ---- decode.cu
int decode_workspace_bytes(const spear_w4_layer& L, int M, size_t* bytes);
int launch_decode(const spear_w4_layer& L, const uint16_t* x, int M, void* y, int out_f32,
                  void* ws, size_t ws_bytes, cudaStream_t st, bool overlap);
int launch_decode_noalloc(const spear_w4_layer& L, const uint16_t* x, int M, void* y, int out_f32,
                          cudaStream_t st);
int read_and_clear_status_decode(unsigned* out, cudaStream_t st);

// ---- decode_ks.cu (cluster K-split decode, 1..32 tokens, no workspace)
bool decode_ks_supports(const spear_w4_layer& L, int M);
int launch_decode_ks(const spear_w4_layer& L, const uint16_t* x, int M, void* y, int out_f32, cudaStream_t st,
                     bool overlap);
int read_and_clear_status_decode_ks(unsigned* out, cudaStream_t st);

// ---- decode_tm.cu (cluster K-split decode on tcgen05, weights in tensor memory, 1..64 tokens)
bool decode_tm_supports(const spear_w4_layer& L, int M);
int launch_decode_tm(const spear_w4_layer& L, const uint16_t* x, int M, void* y, int out_f32, cudaStream_t st,
                     bool overlap);
int read_and_clear_status_decode_tm(unsigned* out, cudaStream_t st);

// ---- decode_tc.cu (tensor-core decode path)
int decode_tc_workspace_bytes(const spear_w4_layer& L, int M, size_t* bytes);
size_t decode_tc_sync_bytes();
int launch_decode_tc(const spear_w4_layer& L, const uint16_t* x, int M, void* y, int out_f32, void* ws,
                     size_t ws_bytes, cudaStream_t st, bool overlap);
int read_and_clear_status_decode_tc(unsigned* out, cudaStream_t st);

// ---- prefill.cu
int prefill_workspace_bytes(const spear_w4_layer& L, int M, int mode, size_t* bytes);
int launch_prefill(const spear_w4_layer& L, const uint16_t* x, int M, void* y, int out_f32,
                   int mode, void* ws, size_t ws_bytes, cudaStream_t st, cudaStream_t st_aux);
int read_and_clear_status_prefill(unsigned* out, cudaStream_t st);

}  // namespace spear
