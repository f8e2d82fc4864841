// api.cu -- the C ABI (include/gdn.h): argument checks and dispatch.
//
// Every argument error is caught here, before any launch, so a rejected call
// writes nothing.  Nothing in this file allocates, frees or synchronises.
#include <cstring>

#include "common.cuh"

namespace {

using namespace gdn;

bool dims_supported(const gdn_problem &p) {
    if (p.head_dim_k != p.head_dim_v) return false;
    if (p.head_dim_k != 64 && p.head_dim_k != 128) return false;
    if (p.qkv_dtype != GDN_BF16 && p.qkv_dtype != GDN_F32) return false;
    return p.num_v_heads % p.num_k_heads == 0;
}

gdn_status check_problem(const gdn_problem *pp) {
    if (!pp) return GDN_ERR_INVALID_ARG;
    const gdn_problem &p = *pp;
    if (p.num_seqs < 0 || p.total_tokens < 0 || p.num_k_heads <= 0 || p.num_v_heads <= 0 ||
        p.head_dim_k <= 0 || p.head_dim_v <= 0)
        return GDN_ERR_INVALID_ARG;
    // Grid dimensions and 32-bit token offsets inside the kernels.
    if (p.total_tokens > (int64_t)INT32_MAX / 2 || p.num_seqs > 65535 ||
        p.num_v_heads > 65535 ||
        (int64_t)p.num_v_heads * p.head_dim_v > (int64_t)1 << 20)
        return GDN_ERR_INVALID_ARG;
    if (!dims_supported(p)) return GDN_ERR_UNSUPPORTED;
    return GDN_OK;
}

bool any_misaligned(std::initializer_list<const void *> ptrs) {
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return true;
    return false;
}

}  // namespace

extern "C" {

GDN_API size_t gdn_chunk_prefill_workspace_size(const gdn_problem *problem) {
    if (check_problem(problem) != GDN_OK) return 0;
    return prefill_tc_supported(*problem) ? prefill_tc_workspace_size(*problem) : 0;
}

}  // extern "C"

namespace {

// The prefill entry points share their checks and dispatch; `snaps` (state
// after every chunk) is only supported on the tensor-core path.
gdn_status prefill_impl(const gdn_problem *problem, const void *q, const void *k, const void *v,
                        const float *g, const float *beta, const int32_t *cu_seqlens,
                        const float *initial_state, void *out, float *final_state, float *snaps,
                        int snap_stride, bool want_snaps, gdn_stream_t stream,
                        int scan_group = -1, void *const *events = nullptr,
                        int *fused = nullptr) {
    const gdn_status st = check_problem(problem);
    if (st != GDN_OK) return st;
    const gdn_problem &p = *problem;
    if ((want_snaps || scan_group >= 0) && !prefill_tc_supported(p)) return GDN_ERR_UNSUPPORTED;
    if (p.num_seqs == 0) return p.total_tokens == 0 ? GDN_OK : GDN_ERR_INVALID_ARG;
    if (!cu_seqlens) return GDN_ERR_INVALID_ARG;
    if (p.total_tokens > 0 && (!q || !k || !v || !g || !beta || !out)) return GDN_ERR_INVALID_ARG;
    if (want_snaps && (!snaps || snap_stride < 1)) return GDN_ERR_INVALID_ARG;
    if (any_misaligned({q, k, v, g, beta, initial_state, out, final_state, snaps}))
        return GDN_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0) return GDN_ERR_MISALIGNED;
    if (out && (out == q || out == k || out == v)) return GDN_ERR_INVALID_ARG;
    if (snaps && (snaps == initial_state || snaps == final_state)) return GDN_ERR_INVALID_ARG;
    if (scan_group == 0) scan_group = prefill_scan_auto_group(p);
    const size_t need = scan_group > 0 ? prefill_scan_workspace_size(p, scan_group)
                                       : gdn_chunk_prefill_workspace_size(problem);
    if (need > 0) {
        if (!p.workspace || p.workspace_bytes < need) return GDN_ERR_WORKSPACE;
        if (!aligned16(p.workspace)) return GDN_ERR_WORKSPACE;
    }
    cudaStream_t st_ = reinterpret_cast<cudaStream_t>(stream);
    if (scan_group > 0) {
        gdn_status st = launch_prefill_scan(p, scan_group, q, k, v, g, beta, cu_seqlens,
                                            initial_state, out, final_state, st_);
        if (kDebug && st == GDN_OK && p.total_tokens > 0)
            st = launch_debug_input_checks(p, q, k, g, beta, static_cast<int *>(p.workspace), st_);
        return st;
    }
    if (prefill_tc_supported(p)) {
        gdn_status st = launch_prefill_tc(p, q, k, v, g, beta, cu_seqlens, initial_state, out,
                                          final_state, snaps, snap_stride, st_, events, fused);
        // (debug builds: the inputs' preconditions, after the call's kernels
        // so that its first kernel's reset of the error word comes before)
        if (kDebug && st == GDN_OK && p.total_tokens > 0)
            st = launch_debug_input_checks(p, q, k, g, beta, static_cast<int *>(p.workspace), st_);
        return st;
    }
    return launch_prefill_simt(p, q, k, v, g, beta, cu_seqlens, initial_state, out, final_state,
                               st_);
}

}  // namespace

extern "C" {

GDN_API gdn_status gdn_chunk_prefill(const gdn_problem *problem, const void *q, const void *k,
                                     const void *v, const float *g, const float *beta,
                                     const int32_t *cu_seqlens, const float *initial_state,
                                     void *out, float *final_state, gdn_stream_t stream) {
    return prefill_impl(problem, q, k, v, g, beta, cu_seqlens, initial_state, out, final_state,
                        nullptr, 1, false, stream);
}

GDN_API int64_t gdn_chunk_prefill_snapshot_slots(const gdn_problem *problem,
                                                 int32_t snapshot_chunks) {
    if (check_problem(problem) != GDN_OK || !prefill_tc_supported(*problem) ||
        snapshot_chunks < 1)
        return 0;
    return prefill_tc_snapshot_slots(*problem, snapshot_chunks);
}

GDN_API gdn_status gdn_chunk_prefill_snapshots(const gdn_problem *problem, const void *q,
                                               const void *k, const void *v, const float *g,
                                               const float *beta, const int32_t *cu_seqlens,
                                               const float *initial_state, void *out,
                                               float *final_state, float *snapshots,
                                               int32_t snapshot_chunks, gdn_stream_t stream) {
    return prefill_impl(problem, q, k, v, g, beta, cu_seqlens, initial_state, out, final_state,
                        snapshots, snapshot_chunks, true, stream);
}

GDN_API size_t gdn_chunk_prefill_scan_workspace_size(const gdn_problem *problem,
                                                    int32_t chunks_per_group) {
    if (check_problem(problem) != GDN_OK || !prefill_tc_supported(*problem) ||
        chunks_per_group < 0)
        return 0;
    const int L = chunks_per_group > 0 ? chunks_per_group : prefill_scan_auto_group(*problem);
    return prefill_scan_workspace_size(*problem, L);
}

GDN_API gdn_status gdn_chunk_prefill_scan(const gdn_problem *problem, int32_t chunks_per_group,
                                          const void *q, const void *k, const void *v,
                                          const float *g, const float *beta,
                                          const int32_t *cu_seqlens, const float *initial_state,
                                          void *out, float *final_state, gdn_stream_t stream) {
    if (chunks_per_group < 0) return GDN_ERR_INVALID_ARG;
    return prefill_impl(problem, q, k, v, g, beta, cu_seqlens, initial_state, out, final_state,
                        nullptr, 1, false, stream, chunks_per_group);
}

GDN_API gdn_status gdn_decode_step(const gdn_problem *problem, const void *q, const void *k,
                                   const void *v, const float *g, const float *beta,
                                   float *state, void *out, gdn_stream_t stream) {
    const gdn_status st = check_problem(problem);
    if (st != GDN_OK) return st;
    const gdn_problem &p = *problem;
    if (p.total_tokens != p.num_seqs) return GDN_ERR_INVALID_ARG;
    if (p.num_seqs == 0) return GDN_OK;
    if (!q || !k || !v || !g || !beta || !state || !out) return GDN_ERR_INVALID_ARG;
    if (any_misaligned({q, k, v, g, beta, state, out})) return GDN_ERR_MISALIGNED;
    if (out == q || out == k || out == v) return GDN_ERR_INVALID_ARG;
    return launch_decode(p, q, k, v, g, beta, state, GDN_F32, out,
                         reinterpret_cast<cudaStream_t>(stream));
}

GDN_API gdn_status gdn_decode_step_half_state(const gdn_problem *problem, const void *q,
                                              const void *k, const void *v, const float *g,
                                              const float *beta, void *state,
                                              int32_t state_dtype, void *out,
                                              gdn_stream_t stream) {
    const gdn_status st = check_problem(problem);
    if (st != GDN_OK) return st;
    const gdn_problem &p = *problem;
    if (p.total_tokens != p.num_seqs) return GDN_ERR_INVALID_ARG;
    if (state_dtype != GDN_F16 && state_dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED;
    if (p.num_seqs == 0) return GDN_OK;
    if (!q || !k || !v || !g || !beta || !state || !out) return GDN_ERR_INVALID_ARG;
    if (any_misaligned({q, k, v, g, beta, state, out})) return GDN_ERR_MISALIGNED;
    if (out == q || out == k || out == v) return GDN_ERR_INVALID_ARG;
    return launch_decode(p, q, k, v, g, beta, state, state_dtype, out,
                         reinterpret_cast<cudaStream_t>(stream));
}

GDN_API gdn_status gdn_verify_step(const gdn_problem *problem, int32_t num_tokens,
                                   const void *q, const void *k, const void *v, const float *g,
                                   const float *beta, const void *state, int32_t state_dtype,
                                   void *slots, void *out, gdn_stream_t stream) {
    const gdn_status st = check_problem(problem);
    if (st != GDN_OK) return st;
    const gdn_problem &p = *problem;
    if (num_tokens < 1 || num_tokens > 8) return GDN_ERR_INVALID_ARG;
    if (p.total_tokens != (int64_t)p.num_seqs * num_tokens) return GDN_ERR_INVALID_ARG;
    if (state_dtype != GDN_F32 && state_dtype != GDN_F16 && state_dtype != GDN_BF16)
        return GDN_ERR_UNSUPPORTED;
    if (p.num_seqs == 0) return GDN_OK;
    if (!q || !k || !v || !g || !beta || !state || !slots || !out) return GDN_ERR_INVALID_ARG;
    if (any_misaligned({q, k, v, g, beta, state, slots, out})) return GDN_ERR_MISALIGNED;
    if (out == q || out == k || out == v || slots == state) return GDN_ERR_INVALID_ARG;
    return launch_verify(p, num_tokens, q, k, v, g, beta, state, state_dtype, slots, out,
                         reinterpret_cast<cudaStream_t>(stream));
}

GDN_API gdn_status gdn_chunk_prefill_device_status(const void *workspace,
                                                   gdn_stream_t stream) {
    const void *ws = workspace ? workspace : gdn::noalloc_scratch();
    if (!ws) return GDN_ERR_CUDA;
    if (!gdn::aligned16(ws)) return GDN_ERR_MISALIGNED;
    int word = 0;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&word, ws, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return GDN_ERR_CUDA;
    switch (word) {
        case gdn::kErrNone: return GDN_OK;
        case gdn::kErrCuSeqlens: return GDN_ERR_INVALID_ARG;
        case gdn::kErrTimeout: return GDN_ERR_TIMEOUT;
        case gdn::kErrInputs: return GDN_ERR_INVALID_ARG;
        case gdn::kErrIndex: return GDN_ERR_INTERNAL;
    }
    return GDN_ERR_CUDA;
}

GDN_API gdn_status gdn_chunk_prefill_timed(const gdn_problem *problem, const void *q,
                                           const void *k, const void *v, const float *g,
                                           const float *beta, const int32_t *cu_seqlens,
                                           const float *initial_state, void *out,
                                           float *final_state, gdn_event_t const *events,
                                           int32_t *fused, gdn_stream_t stream) {
    if (!events || !events[0] || !events[1] || !events[2] || !events[3])
        return GDN_ERR_INVALID_ARG;
    if (fused) *fused = 0;
    const gdn_status st = check_problem(problem);
    if (st != GDN_OK) return st;
    if (!prefill_tc_supported(*problem)) return GDN_ERR_UNSUPPORTED;
    if (problem->num_seqs == 0 && problem->total_tokens == 0) {
        // Nothing to launch: the four events mark the same point.
        const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
        for (int i = 0; i < 4; ++i)
            if (cudaEventRecord(reinterpret_cast<cudaEvent_t>(events[i]), s) != cudaSuccess)
                return GDN_ERR_CUDA;
        return GDN_OK;
    }
    void *ev[4] = {events[0], events[1], events[2], events[3]};
    return prefill_impl(problem, q, k, v, g, beta, cu_seqlens, initial_state, out, final_state,
                        nullptr, 1, false, stream, -1, ev, fused);
}

GDN_API gdn_status gdn_chunk_prefill_prep_only(const gdn_problem *problem, const void *q,
                                               const void *k, const float *g,
                                               const float *beta, const int32_t *cu_seqlens,
                                               gdn_stream_t stream) {
    const gdn_status st = check_problem(problem);
    if (st != GDN_OK) return st;
    const gdn_problem &p = *problem;
    if (!prefill_tc_supported(p)) return GDN_ERR_UNSUPPORTED;
    if (p.num_seqs == 0) return p.total_tokens == 0 ? GDN_OK : GDN_ERR_INVALID_ARG;
    if (!cu_seqlens) return GDN_ERR_INVALID_ARG;
    if (p.total_tokens > 0 && (!q || !k || !g || !beta)) return GDN_ERR_INVALID_ARG;
    if (any_misaligned({q, k, g, beta})) return GDN_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0) return GDN_ERR_MISALIGNED;
    const size_t need = gdn_chunk_prefill_workspace_size(problem);
    if (!p.workspace || p.workspace_bytes < need || !aligned16(p.workspace))
        return GDN_ERR_WORKSPACE;
    return launch_prefill_tc_prep_only(p, q, k, g, beta, cu_seqlens,
                                       reinterpret_cast<cudaStream_t>(stream));
}

GDN_API gdn_status gdn_chunk_prefill_prep_layout(const gdn_problem *problem, int64_t *layout) {
    const gdn_status st = check_problem(problem);
    if (st != GDN_OK) return st;
    if (!layout) return GDN_ERR_INVALID_ARG;
    if (!prefill_tc_supported(*problem)) return GDN_ERR_UNSUPPORTED;
    prefill_tc_slot_layout(*problem, layout);
    return GDN_OK;
}

GDN_API int32_t gdn_prefill_fused_mode(int32_t mode) { return gdn::prefill_fused_mode(mode); }

GDN_API int32_t gdn_prefill_path(const gdn_problem *problem, int32_t sms, int32_t mode) {
    if (check_problem(problem) != GDN_OK || sms < 0 || !gdn::prefill_tc_supported(*problem))
        return -1;
    if (mode < 0 || mode > 3) mode = gdn::prefill_fused_mode(-1);
    return gdn::prefill_path(*problem, sms, sms, mode);
}

GDN_API const char *gdn_status_string(gdn_status status) {
    switch (status) {
        case GDN_OK: return "GDN_OK";
        case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG: invalid argument";
        case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED: configuration not supported";
        case GDN_ERR_MISALIGNED: return "GDN_ERR_MISALIGNED: pointer not 16-byte aligned";
        case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE: workspace missing or too small";
        case GDN_ERR_CUDA: return "GDN_ERR_CUDA: CUDA launch or runtime error";
        case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT: a bounded wait inside a kernel ran out";
        case GDN_ERR_INTERNAL:
            return "GDN_ERR_INTERNAL: a device-side index check of a debug build failed";
    }
    return "GDN_ERR_UNKNOWN";
}

GDN_API int gdn_version(void) { return 100; }

}  // extern "C"
