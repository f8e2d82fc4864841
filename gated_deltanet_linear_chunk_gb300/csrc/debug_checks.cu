// debug_checks.cu -- GDN_DEBUG builds only: the documented preconditions of a
// prefill's inputs, checked on the device after the call's kernels (the
// compute sanitizer being unavailable, debug builds check what they can
// themselves).  A violation records kErrInputs in the workspace error word,
// which gdn_chunk_prefill_device_status reports as GDN_ERR_INVALID_ARG.
//
// Checked: every g finite and <= 0; every beta in [0, 1]; every q and k row
// (one token, one key head) of unit L2 norm within kNormTol, the rounding
// of a row normalised in higher precision and stored in bf16.
#include <math.h>

#include "common.cuh"

namespace gdn {
namespace {

constexpr float kNormTol = 1e-2f;
constexpr int kCheckThreads = 256;

template <typename TIn>
__global__ void __launch_bounds__(kCheckThreads)
gdn_debug_input_check_kernel(const TIn *__restrict__ q, const TIn *__restrict__ k,
                             const float *__restrict__ g, const float *__restrict__ beta,
                             int64_t T, int Hk, int Hv, int dk, int *__restrict__ err) {
    const int lane = threadIdx.x & 31;
    const int64_t n_threads = (int64_t)gridDim.x * blockDim.x;
    const int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    // q and k rows: one warp per (token, key head).
    for (int64_t r = t0 / 32; r < T * Hk; r += n_threads / 32) {
        float sq = 0.f, sk = 0.f;
        for (int e = lane; e < dk; e += 32) {
            const float a = to_f32(q[r * dk + e]), b = to_f32(k[r * dk + e]);
            sq = fmaf(a, a, sq);
            sk = fmaf(b, b, sk);
        }
        sq = warp_sum(sq);
        sk = warp_sum(sk);
        if (lane == 0 && !(fabsf(sqrtf(sq) - 1.f) <= kNormTol && fabsf(sqrtf(sk) - 1.f) <= kNormTol))
            debug_fail(err, kErrInputs);
    }
    // g and beta, element by element (comparisons false on NaN).
    for (int64_t i = t0; i < T * Hv; i += n_threads) {
        const float gv = g[i], bv = beta[i];
        if (!(isfinite(gv) && gv <= 0.f) || !(bv >= 0.f && bv <= 1.f))
            debug_fail(err, kErrInputs);
    }
}

}  // namespace

gdn_status launch_debug_input_checks(const gdn_problem &p, const void *q, const void *k,
                                     const float *g, const float *beta, int *err,
                                     cudaStream_t stream) {
    if (!err || p.total_tokens == 0) return GDN_OK;
    const int64_t rows = p.total_tokens * p.num_k_heads;
    const int64_t want = (rows * 32 + kCheckThreads - 1) / kCheckThreads;
    const unsigned blocks = (unsigned)(want < 1216 ? (want > 0 ? want : 1) : 1216);
    if (p.qkv_dtype == GDN_BF16)
        gdn_debug_input_check_kernel<__nv_bfloat16><<<blocks, kCheckThreads, 0, stream>>>(
            static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k), g,
            beta, p.total_tokens, p.num_k_heads, p.num_v_heads, p.head_dim_k, err);
    else
        gdn_debug_input_check_kernel<float><<<blocks, kCheckThreads, 0, stream>>>(
            static_cast<const float *>(q), static_cast<const float *>(k), g, beta,
            p.total_tokens, p.num_k_heads, p.num_v_heads, p.head_dim_k, err);
    return launch_status();
}

}  // namespace gdn
