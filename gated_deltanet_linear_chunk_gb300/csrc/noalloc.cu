// noalloc.cu -- gdn_chunk_prefill_noalloc: the chunked prefill with its
// scratch memory built into the library instead of passed in by the caller.
//
// Some callers cannot allocate device memory when they call the layer:
// serving engines that reserve nearly all device memory for their own pools
// at start-up, plug-ins that run inside a host framework which owns the
// allocator, and latency-critical paths where cudaMalloc (which may
// synchronise the whole device) is not acceptable.  For them this entry
// point takes its scratch from one fixed array in device memory that every
// GPU loading this library holds until the process exits.
//
// Contract of the array:
//  * at most kScratchBytes (64 MiB); larger problems are rejected with
//    GDN_ERR_WORKSPACE before anything is launched;
//  * every call shares it and it keeps the previous call's contents; the
//    kernels rewrite every byte they read before reading it (the chunk table
//    and the error word are rebuilt at the start of each call), so no
//    clearing is needed between calls;
//  * two calls whose work overlaps on the GPU (different streams, no
//    ordering between them) race on the array: order such calls.
//
// In host code the array's name only stands in for the symbol; its device
// address comes from cudaGetSymbolAddress, looked up once per device, on the
// first call made with that device current.  Make that first call before
// any stream capture.
#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kScratchBytes = size_t(64) << 20;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch for the current device (nullptr on failure).
void *scratch_for_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = ptr;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

namespace gdn {
void *noalloc_scratch() { return scratch_for_current_device(); }
}  // namespace gdn

extern "C" {

GDN_API gdn_status gdn_chunk_prefill_noalloc(const gdn_problem *problem, const void *q,
                                             const void *k, const void *v, const float *g,
                                             const float *beta, const int32_t *cu_seqlens,
                                             const float *initial_state, void *out,
                                             float *final_state, gdn_stream_t stream) {
    if (!problem) return GDN_ERR_INVALID_ARG;
    gdn_problem p = *problem;
    p.workspace = nullptr;
    p.workspace_bytes = 0;
    const size_t need = gdn_chunk_prefill_workspace_size(&p);
    if (need > kScratchBytes) return GDN_ERR_WORKSPACE;
    if (need > 0) {
        void *ptr = scratch_for_current_device();
        if (!ptr) return GDN_ERR_CUDA;
        p.workspace = ptr;
        p.workspace_bytes = kScratchBytes;
    }
    return gdn_chunk_prefill(&p, q, k, v, g, beta, cu_seqlens, initial_state, out, final_state,
                             stream);
}

}  // extern "C"
