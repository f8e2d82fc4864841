// host_pipeline.cu -- gdn_chunk_prefill_host: one sequence's prefill from
// host memory, with the transfers overlapped with the computation.
//
// The sequence is cut into pieces of whole 64-token chunks, the last two
// smaller than the others.  Piece p's inputs go up on an upload stream while
// piece p - 1 is computed on the caller's stream.  Its output comes back on
// a download stream while piece p + 1 is computed.  The pieces are chained through a device state buffer
// (each piece's final state is the next one's initial state), which is
// exactly the whole prefill, because chunks restart at every 64 tokens.
// Besides the prefill kernels this issues only cudaMemcpyAsync,
// cudaMemsetAsync and event operations.
#include <algorithm>
#include <mutex>

#include "common.cuh"

namespace {

using namespace gdn;

constexpr int kMaxPieces = 64;
constexpr int kMaxDevices = 64;

// Streams and events of the pipeline, one set per device, created at that
// device's first call (non-blocking streams; events without timing).  Calls
// on one device hold its mutex while they issue their work, so concurrent
// callers never re-record an event another call is still about to wait on;
// a wait takes the event as it stands when the wait is issued, so the next
// call may re-record it at once.
struct Pipe {
    cudaStream_t up = nullptr, down = nullptr;
    cudaEvent_t start = nullptr, up_done[kMaxPieces] = {}, comp_done[kMaxPieces] = {},
                down_done = nullptr;
    bool ok = false;
    std::once_flag once;
    std::mutex mu;
};

Pipe g_pipes[kMaxDevices];

// The current device's pipeline, or nullptr if it cannot be created.
Pipe *pipe() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    Pipe &p = g_pipes[dev];
    std::call_once(p.once, [&p] {
        bool ok = cudaStreamCreateWithFlags(&p.up, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&p.down, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaEventCreateWithFlags(&p.start, cudaEventDisableTiming) == cudaSuccess &&
                  cudaEventCreateWithFlags(&p.down_done, cudaEventDisableTiming) == cudaSuccess;
        for (int i = 0; ok && i < kMaxPieces; ++i)
            ok = cudaEventCreateWithFlags(&p.up_done[i], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&p.comp_done[i], cudaEventDisableTiming) == cudaSuccess;
        p.ok = ok;
    });
    return p.ok ? &p : nullptr;
}

struct PieceLens {
    int32_t len[kMaxPieces];
};

// cu[2 i], cu[2 i + 1] = 0, length of piece i: each piece's cu_seqlens.
__global__ void gdn_piece_cu_kernel(int32_t *cu, PieceLens lens, int pieces) {
    for (int i = threadIdx.x; i < pieces; i += blockDim.x) {
        cu[2 * i] = 0;
        cu[2 * i + 1] = lens.len[i];
    }
}

}  // namespace

extern "C" {

GDN_API gdn_status gdn_chunk_prefill_host(
    const gdn_problem *problem, int32_t pieces, const void *q_h, const void *k_h, const void *v_h,
    const float *g_h, const float *beta_h, void *out_h, const float *initial_state,
    float *final_state, void *q_d, void *k_d, void *v_d, float *g_d, float *beta_d, void *out_d,
    int32_t *cu_d, float *state_d, gdn_stream_t stream) {
    if (!problem) return GDN_ERR_INVALID_ARG;
    const gdn_problem &p = *problem;
    if (p.num_seqs != 1 || p.total_tokens < 0 || pieces < 1 || pieces > kMaxPieces)
        return GDN_ERR_INVALID_ARG;
    if (p.qkv_dtype != GDN_BF16 && p.qkv_dtype != GDN_F32) return GDN_ERR_UNSUPPORTED;
    const int64_t T = p.total_tokens;
    if (T > 0 && (!q_h || !k_h || !v_h || !g_h || !beta_h || !out_h || !q_d || !k_d || !v_d ||
                  !g_d || !beta_d || !out_d))
        return GDN_ERR_INVALID_ARG;
    if (!cu_d || !state_d) return GDN_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(state_d) % 16 || reinterpret_cast<uintptr_t>(cu_d) % 16)
        return GDN_ERR_MISALIGNED;
    const size_t el = p.qkv_dtype == GDN_BF16 ? 2 : 4;
    const size_t qk_row = (size_t)p.num_k_heads * p.head_dim_k * el;
    const size_t v_row = (size_t)p.num_v_heads * p.head_dim_v * el;
    const size_t gb_row = (size_t)p.num_v_heads * 4;
    const size_t state_bytes = (size_t)p.num_v_heads * p.head_dim_v * p.head_dim_k * 4;
    // The whole sequence's workspace covers every piece: check it before
    // anything is enqueued.
    const size_t need = gdn_chunk_prefill_workspace_size(&p);
    if (need > 0 && (!p.workspace || p.workspace_bytes < need)) return GDN_ERR_WORKSPACE;
    Pipe *ppp = pipe();
    if (!ppp) return GDN_ERR_CUDA;
    Pipe &pp = *ppp;
    std::lock_guard<std::mutex> lock(pp.mu);
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);

    // Piece boundaries at whole chunks: equal shares, except that the last
    // two pieces (of three or more; the last of two) get a half and a
    // quarter of a share.  What is left after the last upload (that piece's
    // computation and download) is then short, and the link, which carries
    // the other pieces' downloads beside the uploads, stays busy.  Every
    // piece gets at least one chunk.
    const int64_t chunks = (T + 63) / 64;
    if (pieces > chunks) pieces = (int32_t)(chunks > 0 ? chunks : 1);
    int64_t bnd[kMaxPieces + 1];
    PieceLens lens;
    {
        int64_t w[kMaxPieces], total = 0;
        for (int i = 0; i < pieces; ++i)
            w[i] = pieces >= 3 ? (i < pieces - 2 ? 4 : i == pieces - 2 ? 2 : 1)
                               : (pieces == 2 ? (i == 0 ? 2 : 1) : 1);
        for (int i = 0; i < pieces; ++i) total += w[i];
        int64_t acc = 0, c_prev = 0;
        bnd[0] = 0;
        for (int i = 1; i <= pieces; ++i) {
            acc += w[i - 1];
            const int64_t c = std::min<int64_t>(std::max<int64_t>((chunks * acc) / total, c_prev + 1),
                                                chunks - (pieces - i));
            bnd[i] = std::min<int64_t>(T, 64 * c);
            c_prev = c;
        }
    }
    for (int i = 0; i < pieces; ++i) lens.len[i] = (int32_t)(bnd[i + 1] - bnd[i]);

    // The state chain starts from the initial state (or zero).
    if (initial_state) {
        if (cudaMemcpyAsync(state_d, initial_state, state_bytes, cudaMemcpyDeviceToDevice, cs) !=
            cudaSuccess)
            return GDN_ERR_CUDA;
    } else if (cudaMemsetAsync(state_d, 0, state_bytes, cs) != cudaSuccess) {
        return GDN_ERR_CUDA;
    }
    gdn_piece_cu_kernel<<<1, 64, 0, cs>>>(cu_d, lens, pieces);
    if (cudaGetLastError() != cudaSuccess || cudaEventRecord(pp.start, cs) != cudaSuccess ||
        cudaStreamWaitEvent(pp.up, pp.start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(pp.down, pp.start, 0) != cudaSuccess)
        return GDN_ERR_CUDA;

    // After an error, the caller's stream still waits for whatever the upload
    // and download streams already hold, so no copy outlives the call's
    // ordering (best effort: the first error is the one returned).
    auto fail = [&](gdn_status st) {
        if (cudaEventRecord(pp.up_done[0], pp.up) == cudaSuccess)
            cudaStreamWaitEvent(cs, pp.up_done[0], 0);
        if (cudaEventRecord(pp.down_done, pp.down) == cudaSuccess)
            cudaStreamWaitEvent(cs, pp.down_done, 0);
        return st;
    };
    auto up = [&](void *dst, const void *src, size_t row, int i) {
        const size_t off = (size_t)bnd[i] * row, n = (size_t)lens.len[i] * row;
        return n == 0 || cudaMemcpyAsync(static_cast<uint8_t *>(dst) + off,
                                         static_cast<const uint8_t *>(src) + off, n,
                                         cudaMemcpyHostToDevice, pp.up) == cudaSuccess;
    };
    for (int i = 0; i < pieces; ++i) {
        if (!up(q_d, q_h, qk_row, i) || !up(k_d, k_h, qk_row, i) || !up(v_d, v_h, v_row, i) ||
            !up(g_d, g_h, gb_row, i) || !up(beta_d, beta_h, gb_row, i) ||
            cudaEventRecord(pp.up_done[i], pp.up) != cudaSuccess)
            return fail(GDN_ERR_CUDA);
    }
    for (int i = 0; i < pieces; ++i) {
        if (cudaStreamWaitEvent(cs, pp.up_done[i], 0) != cudaSuccess) return fail(GDN_ERR_CUDA);
        gdn_problem pi = p;
        pi.total_tokens = lens.len[i];
        const size_t o = (size_t)bnd[i];
        const gdn_status st = gdn_chunk_prefill(
            &pi, static_cast<const uint8_t *>(q_d) + o * qk_row,
            static_cast<const uint8_t *>(k_d) + o * qk_row,
            static_cast<const uint8_t *>(v_d) + o * v_row, g_d + o * p.num_v_heads,
            beta_d + o * p.num_v_heads, cu_d + 2 * i, state_d,
            static_cast<uint8_t *>(out_d) + o * v_row, state_d, stream);
        if (st != GDN_OK) return fail(st);
        if (cudaEventRecord(pp.comp_done[i], cs) != cudaSuccess ||
            cudaStreamWaitEvent(pp.down, pp.comp_done[i], 0) != cudaSuccess)
            return fail(GDN_ERR_CUDA);
        const size_t n = (size_t)lens.len[i] * v_row;
        if (n && cudaMemcpyAsync(static_cast<uint8_t *>(out_h) + o * v_row,
                                 static_cast<const uint8_t *>(out_d) + o * v_row, n,
                                 cudaMemcpyDeviceToHost, pp.down) != cudaSuccess)
            return fail(GDN_ERR_CUDA);
    }
    if (final_state && cudaMemcpyAsync(final_state, state_d, state_bytes,
                                       cudaMemcpyDeviceToDevice, cs) != cudaSuccess)
        return fail(GDN_ERR_CUDA);
    if (cudaEventRecord(pp.down_done, pp.down) != cudaSuccess ||
        cudaStreamWaitEvent(cs, pp.down_done, 0) != cudaSuccess)
        return GDN_ERR_CUDA;
    return GDN_OK;
}

}  // extern "C"
