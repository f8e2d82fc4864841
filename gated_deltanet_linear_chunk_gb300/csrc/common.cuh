// common.cuh -- small shared helpers of the CUDA library (not part of the ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

// Load one element of an input tensor as fp32.
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// Store an fp32 value in the output dtype (bf16: round to nearest even).
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Error word at offset 0 of the tensor-core prefill's workspace, written by
// its kernels (reset by the first kernel of every call).  The last two only
// by GDN_DEBUG builds: kErrInputs for inputs outside the documented
// preconditions, kErrIndex for a failed internal index check (a bug).
enum DeviceError : int {
    kErrNone = 0,
    kErrCuSeqlens = 1,
    kErrTimeout = 2,
    kErrInputs = 3,
    kErrIndex = 4
};

// GDN_DEBUG builds check, on the device, the inputs' documented
// preconditions and the kernels' table-derived indices: a failed check
// records its code in the error word (the first one wins) and the access it
// guards is skipped; nothing traps.
#ifdef GDN_DEBUG
constexpr bool kDebug = true;
#else
constexpr bool kDebug = false;
#endif

__device__ __forceinline__ void debug_fail(int *err, int code) {
    if (err) atomicCAS(err, (int)kErrNone, code);
}

// Launch helpers return a gdn_status for the last launch on this thread.
inline gdn_status launch_status() {
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

// Kernel launchers implemented in the .cu files.
// Verify step: num_tokens (1..8) tokens per sequence from `state`, the state
// after token t in slot t (storage state_dtype for both).
gdn_status launch_verify(const gdn_problem &p, int num_tokens, const void *q, const void *k,
                         const void *v, const float *g, const float *beta, const void *state,
                         int state_dtype, void *slots, void *out, cudaStream_t stream);
// state_dtype: GDN_F32, GDN_F16 or GDN_BF16 (storage of the state).
gdn_status launch_decode(const gdn_problem &p, const void *q, const void *k, const void *v,
                         const float *g, const float *beta, void *state, int state_dtype,
                         void *out, cudaStream_t stream);
gdn_status launch_prefill_simt(const gdn_problem &p, const void *q, const void *k,
                               const void *v, const float *g, const float *beta,
                               const int32_t *cu_seqlens, const float *h0, void *out,
                               float *hT, cudaStream_t stream);

// GDN_DEBUG builds: checks of a prefill's inputs on `stream` (g <= 0, beta in
// [0, 1], unit-norm q and k rows; all finite), kErrInputs into *err on a
// failure.
gdn_status launch_debug_input_checks(const gdn_problem &p, const void *q, const void *k,
                                     const float *g, const float *beta, int *err,
                                     cudaStream_t stream);

// Device address of the no-alloc entry point's built-in scratch on the
// current device (nullptr if it cannot be looked up).
void *noalloc_scratch();

size_t prefill_tc_workspace_size(const gdn_problem &p);
bool prefill_tc_supported(const gdn_problem &p);
// snaps: fp32 [slots, Hv, dv, dk] or nullptr: the state after every
// snap_stride-th chunk and after the last chunk of every sequence.
// Chunk-parallel scan of the tensor-core prefill (chunks_per_group >= 1).
size_t prefill_scan_workspace_size(const gdn_problem &p, int chunks_per_group);
int prefill_scan_auto_group(const gdn_problem &p);
gdn_status launch_prefill_scan(const gdn_problem &p, int chunks_per_group, const void *q,
                               const void *k, const void *v, const float *g, const float *beta,
                               const int32_t *cu, const float *h0, void *out, float *hT,
                               cudaStream_t stream);

// Fused prep + recurrence mode: sets it (0, 1, 2, 3) and returns the old one;
// any other value only queries.
int prefill_fused_mode(int mode);

// The kernels a tensor-core prefill of `p` runs in fused mode `mode`, with
// the fused kernels' variants able to use `grid` and `grid_m` SMs (0: not at
// all): 0 separate prep and recurrence, 1 fused, 2 fused with one recurrence
// per value head.
int prefill_path(const gdn_problem &p, int grid, int grid_m, int mode);

// events: null, or four caller-created events recorded on `stream` before
// the chunk table, after it, after prep and after the recurrence; *fused
// (if given) is set to whether prep and the recurrence ran as one launch.
gdn_status launch_prefill_tc(const gdn_problem &p, const void *q, const void *k, const void *v,
                             const float *g, const float *beta, const int32_t *cu_seqlens,
                             const float *h0, void *out, float *hT, float *snaps,
                             int snap_stride, cudaStream_t stream, void *const *events = nullptr,
                             int *fused = nullptr);
// Chunk table and prep only (diagnostics), and where prep's products lie in
// the workspace: {slot array offset, slot bytes, W^T, T diag(b), P,
// diag(e^gamma) Q, e^gamma, e^{gamma_L - gamma} offsets within a slot}.
gdn_status launch_prefill_tc_prep_only(const gdn_problem &p, const void *q, const void *k,
                                      const float *g, const float *beta, const int32_t *cu,
                                      cudaStream_t stream);
void prefill_tc_slot_layout(const gdn_problem &p, int64_t *layout);
// Snapshot slots of a problem with one snapshot per snap_stride chunks (a
// bound on the batch's count).
int64_t prefill_tc_snapshot_slots(const gdn_problem &p, int snap_stride);

}  // namespace gdn
