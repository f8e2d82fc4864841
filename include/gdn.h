/*
 * gdn.h -- C ABI of the GB300 (sm_103a) Gated DeltaNet layer library.
 *
 * The layer: for every sequence n and value head h (key head hk = h / (Hv/Hk),
 * contiguous groups), a dv x dk fp32 state S evolves token by token as
 *
 *     S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T,   a_t = exp(g_t),
 *     o_t = S_t q_t                       (updated state, no 1/sqrt(d) scale)
 *
 * with L2-normalised q and k, g <= 0 and b in [0, 1].  Source: the Gated
 * DeltaNet linear-attention layers that make up 48 of the 64 layers of the
 * hybrid Qwen3.8-27B model; page "cf-1.com", section "三个优化", item 2
 * ("GDN prefill": chunk length 64; intra-chunk prep, inter-chunk state
 * recurrence and output), and page "reactapp.top", section "Exploiter
 * l'architecture hybride" (fixed-size state per conversation, fp32, about
 * 150 MB per request over 48 layers = 48 value heads x 128 x 128 x 4 B each).
 *
 * Layouts (row-major, token-major, sequences packed back to back):
 *   q, k          [T, Hk, dk]       qkv dtype (bf16 or fp32)
 *   v, out        [T, Hv, dv]       qkv dtype
 *   g, beta       [T, Hv]           fp32
 *   cu_seqlens    [N + 1]           int32, device memory
 *   state         [N, Hv, dv, dk]   fp32; row i is value dimension i,
 *                                   contiguous over the dk key dimensions
 * All pointers are DEVICE pointers unless stated otherwise.
 *
 * Ownership and threading: the caller owns every buffer.  The library never
 * allocates device memory, never frees, never synchronises, and launches only
 * on the given stream.  Calls are reentrant.  The process-wide state is:
 *   - per device, an attribute cache (SM count, whether each variant of the
 *     fused prefill kernel fits and its launch attribute, the resident CTAs
 *     of the persistent decode kernels and their shared-memory attribute),
 *     filled once per device and kernel under a lock;
 *   - the fused-path mode of gdn_prefill_fused_mode (an atomic integer);
 *   - per device, the upload and download streams of gdn_chunk_prefill_host
 *     (created at its first call on that device);
 *   - per device, the address of gdn_chunk_prefill_noalloc's built-in
 *     scratch array.
 *
 * Errors: argument errors are detected on the host before any launch and
 * leave every output untouched.  Launch failures return GDN_ERR_CUDA.  Faults
 * inside a kernel surface asynchronously at the caller's next
 * synchronisation, as for any CUDA launch.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define GDN_API __attribute__((visibility("default")))
#else
#define GDN_API
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *gdn_stream_t;

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1,  /* null pointer, negative size, inconsistent sizes */
    GDN_ERR_UNSUPPORTED = 2,  /* head dims, head grouping or dtype not built   */
    GDN_ERR_MISALIGNED = 3,   /* a tensor pointer is not 16-byte aligned       */
    GDN_ERR_WORKSPACE = 4,    /* workspace missing, too small or misaligned    */
    GDN_ERR_CUDA = 5,         /* a CUDA runtime call or launch failed          */
    GDN_ERR_TIMEOUT = 6,      /* a bounded wait inside a kernel ran out
                                 (reported by gdn_chunk_prefill_device_status) */
    GDN_ERR_INTERNAL = 7      /* a device-side index check of a GDN_DEBUG build
                                 failed (reported likewise; a library bug) */
} gdn_status;

typedef enum {
    GDN_BF16 = 0,  /* q, k, v and out are bf16 (tensor-core path)   */
    GDN_F32 = 1,   /* q, k, v and out are fp32 (FFMA check path)    */
    GDN_F16 = 2    /* only as the state storage of
                      gdn_decode_step_half_state                    */
} gdn_dtype;

/*
 * Problem descriptor shared by every entry point.
 *   num_seqs      N >= 0 sequences (decode: the batch, one token each)
 *   total_tokens  T = cu_seqlens[N] (prefill); must equal N for decode
 *   num_k_heads   Hk >= 1;  num_v_heads Hv, a multiple of Hk
 *   head_dim_k    dk, head_dim_v dv: 64 or 128, dk == dv
 *   qkv_dtype     a gdn_dtype
 *   workspace     device scratch for the prefill (see the size query);
 *                 16-byte aligned; ignored by the decode step
 */
typedef struct {
    int32_t num_seqs;
    int64_t total_tokens;
    int32_t num_k_heads;
    int32_t num_v_heads;
    int32_t head_dim_k;
    int32_t head_dim_v;
    int32_t qkv_dtype;
    void *workspace;
    size_t workspace_bytes;
} gdn_problem;

/*
 * Bytes of device workspace gdn_chunk_prefill needs for this problem (it
 * depends on N, T, Hk, Hv, the head dims and the dtype).  Returns 0 when the
 * descriptor is invalid or the configuration needs no workspace.
 */
GDN_API size_t gdn_chunk_prefill_workspace_size(const gdn_problem *problem);

/*
 * Chunked prefill (chunk length 64) over N packed sequences.
 *   q, k, v        inputs as laid out above (qkv dtype)
 *   g, beta        fp32 log-decay (<= 0) and write strength per token and
 *                  value head
 *   cu_seqlens     device int32 [N + 1]: cu[0] = 0, nondecreasing, cu[N] = T.
 *                  Zero-length sequences are allowed (their final state is
 *                  the initial state).  Not checked on the host.
 *   initial_state  fp32 [N, Hv, dv, dk] or NULL (zero start)
 *   out            [T, Hv, dv], qkv dtype; must not alias any input
 *   final_state    fp32 [N, Hv, dv, dk] or NULL (not written); may equal
 *                  initial_state (in-place resume)
 * q and k must already be L2-normalised by the caller.  All tensor pointers
 * must be 16-byte aligned.
 *
 * For bf16 and dk = dv = 128, when the N x Hv recurrences leave at least 16
 * SMs free, the intra-chunk prep and the recurrence run as one cooperative
 * launch: prep on the free SMs, publishing each chunk as it is done (every
 * sequence's chunk c before any chunk c + 1), and the recurrences following
 * (each first preps its own first four chunks).  When they do not, the
 * fused launch can instead run Hv recurrences, each taking one value head
 * through every sequence in turn (restarting from each sequence's initial
 * state), with prep publishing the chunks in their packed order.  Otherwise
 * prep and the recurrence are separate kernels.  The results are the same
 * every way.  By default either fused variant is used when a cost model of
 * the paths expects it to be faster: the first for long sequences with few
 * (sequence, value head) pairs, the per-head one for batches whose
 * recurrences would run in several waves; see gdn_prefill_fused_mode.
 */
GDN_API gdn_status gdn_chunk_prefill(const gdn_problem *problem,
                                     const void *q, const void *k, const void *v,
                                     const float *g, const float *beta,
                                     const int32_t *cu_seqlens,
                                     const float *initial_state,
                                     void *out, float *final_state,
                                     gdn_stream_t stream);

/*
 * gdn_chunk_prefill of ONE sequence from HOST memory, with the transfers
 * overlapped with the computation.
 *
 * The sequence is cut into `pieces` pieces of whole 64-token chunks; the
 * output is that of one gdn_chunk_prefill, because chunks restart every 64
 * tokens and each piece starts from the previous piece's state.  The pieces
 * take equal shares of the chunks, except the last two (of three or more),
 * which take a half and a quarter of a share (of two pieces, the second
 * takes half the first's), so that little computation and download is left
 * once the last upload ends; every piece has at least one chunk.  Piece p's
 * inputs are copied up on an upload stream while piece p - 1 is computed on
 * `stream`, and its output is copied back on a download stream while piece
 * p + 1 is computed.  Overlapping the link's two directions with the
 * computation is how a host-resident prompt reaches the GPU fastest.
 *
 * Host buffers (pinned, or the copies do not overlap; layouts as above):
 *   q_h, k_h, v_h, g_h, beta_h   inputs, read
 *   out_h                        output, written
 * Device buffers:
 *   initial_state, final_state   as in gdn_chunk_prefill (NULL allowed)
 *   q_d, k_d, v_d, g_d, beta_d, out_d   staging, full size, as the
 *                                device tensors of gdn_chunk_prefill
 *   cu_d                         scratch int32 [128], 16-byte aligned
 *   state_d                      scratch fp32 [Hv, dv, dk], 16-byte aligned
 *   problem->workspace           as for gdn_chunk_prefill of the whole problem
 * Arguments:
 *   problem   num_seqs must be 1
 *   pieces    1-64; fewer when the sequence has fewer chunks
 *
 * On return everything is enqueued; `stream` completes after the last
 * output byte is back in out_h.  Each device has one upload and one download
 * stream with their events, created at the first call on that device (the
 * current device); calls on one device from several host threads take turns
 * while they enqueue, and their transfers share those two streams.
 * Returns GDN_ERR_INVALID_ARG for num_seqs != 1, a pieces value out of range
 * or a missing buffer; otherwise the errors of gdn_chunk_prefill.
 */
GDN_API gdn_status gdn_chunk_prefill_host(
    const gdn_problem *problem, int32_t pieces, const void *q_h, const void *k_h,
    const void *v_h, const float *g_h, const float *beta_h, void *out_h,
    const float *initial_state, float *final_state, void *q_d, void *k_d, void *v_d, float *g_d,
    float *beta_d, void *out_d, int32_t *cu_d, float *state_d, gdn_stream_t stream);

/*
 * Snapshot slots gdn_chunk_prefill_snapshots needs for this problem with
 * one snapshot every snapshot_chunks chunks: ceil((ceil(T / 64) + N) /
 * snapshot_chunks) + N, a bound on the batch's count (sum over sequences of
 * ceil(chunks_n / snapshot_chunks)).  0 when the descriptor is invalid,
 * snapshot_chunks < 1, or the configuration has no snapshot support.
 */
GDN_API int64_t gdn_chunk_prefill_snapshot_slots(const gdn_problem *problem,
                                                 int32_t snapshot_chunks);

/*
 * gdn_chunk_prefill that also writes the state at chunk boundaries of every
 * sequence, for prefix caching (page "reactapp.top", section "Pourquoi cela
 * convient aux agents harness": the prefix cache keeps the DeltaNet
 * recurrent state, not only the attention KV data; page "note.hsfp.cn",
 * section "5. 三级缓存体系": cached prefix states are restored and only the
 * rest of the prompt is prefilled).
 *   snapshot_chunks  s >= 1: a snapshot after chunks s - 1, 2 s - 1, ... of
 *              each sequence (every 64 s tokens) and after its last chunk
 *   snapshots  fp32 [slots, Hv, dv, dk] (slots from the query above).
 *              Sequence n owns slots base_n .. base_n + ceil(chunks_n / s) - 1,
 *              base_n = sum_{m<n} ceil(chunks_m / s), chunks_n =
 *              ceil(len_n / 64); its slot base_n + i holds the state after
 *              token min(64 s (i + 1), len_n), ready to be passed back as an
 *              initial state.  Slots past the batch's count are not written.
 *              Must not alias the states.
 * Only for bf16 q/k/v with dk = dv = 128 (the tensor-core path); other
 * configurations return GDN_ERR_UNSUPPORTED.  Everything else as
 * gdn_chunk_prefill (same workspace size).  The states are staged in shared
 * memory and stored by TMA after each selected chunk: at 4000 tokens x 48
 * heads, s = 1 costs about half a plain call more, s = 8 (512 tokens) about
 * a tenth.
 */
GDN_API gdn_status gdn_chunk_prefill_snapshots(const gdn_problem *problem,
                                               const void *q, const void *k, const void *v,
                                               const float *g, const float *beta,
                                               const int32_t *cu_seqlens,
                                               const float *initial_state,
                                               void *out, float *final_state,
                                               float *snapshots, int32_t snapshot_chunks,
                                               gdn_stream_t stream);

/*
 * gdn_chunk_prefill with the chunk recurrence run as a chunk-parallel scan,
 * for batches with few (sequence, value head) pairs and long sequences.
 *
 * The chunk step of a head is affine in the state, S_{c+1} = S_c M_c + B_c.
 * That is a restatement of the chunk recurrence of the pages (page
 * "cf-1.com", section "三个优化", item 2: the inter-chunk state propagation
 * is the sequential part that dominates the layer's time).  Steps:
 *   1. Each sequence is cut into groups of chunks_per_group chunks.
 *   2. Every group's composite (M, B) is computed in parallel: B is the
 *      recurrence from a zero state, M the recurrence of the linear part
 *      from the identity.
 *   3. The state is carried across groups in fp32.
 *   4. The outputs of every group are produced in parallel from the state
 *      entering it.
 * Results are those of gdn_chunk_prefill up to rounding order.
 *
 *   chunks_per_group  >= 1 chunks (64 tokens each) per group, or 0 to choose
 *              one so that groups x value heads about fills the GPU's SMs
 *   problem->workspace, workspace_bytes: at least
 *              gdn_chunk_prefill_scan_workspace_size(problem, chunks_per_group)
 *   everything else as gdn_chunk_prefill
 *
 * Only for bf16 q/k/v with dk = dv = 128.  Other configurations return
 * GDN_ERR_UNSUPPORTED, and the size query returns 0 for them.  The query
 * also returns 0 for an invalid descriptor or chunks_per_group < 0; the call
 * returns GDN_ERR_INVALID_ARG for chunks_per_group < 0.
 */
GDN_API size_t gdn_chunk_prefill_scan_workspace_size(const gdn_problem *problem,
                                                    int32_t chunks_per_group);
GDN_API gdn_status gdn_chunk_prefill_scan(const gdn_problem *problem, int32_t chunks_per_group,
                                          const void *q, const void *k, const void *v,
                                          const float *g, const float *beta,
                                          const int32_t *cu_seqlens, const float *initial_state,
                                          void *out, float *final_state, gdn_stream_t stream);

/*
 * One recurrent decode step for N sequences (one token each), updating the
 * state in place:
 *   q, k   [N, Hk, dk];  v, out [N, Hv, dv] (qkv dtype);  g, beta [N, Hv] fp32
 *   state  fp32 [N, Hv, dv, dk], read and written in place
 * problem->total_tokens must equal problem->num_seqs.
 */
GDN_API gdn_status gdn_decode_step(const gdn_problem *problem,
                                   const void *q, const void *k, const void *v,
                                   const float *g, const float *beta,
                                   float *state, void *out,
                                   gdn_stream_t stream);

/*
 * gdn_decode_step with the state stored in 16 bits: each step reads the
 * stored state, computes in fp32 exactly as gdn_decode_step does and stores
 * the updated state rounded to nearest even, halving the state traffic that
 * bounds the step.  (Page "reactapp.top", section "Exploiter l'architecture
 * hybride": the forked server keeps this state in fp16 instead of fp32, at
 * perplexity unchanged to three decimals.)
 *   state        [N, Hv, dv, dk] in state_dtype, read and written in place
 *   state_dtype  GDN_F16 (the pages' choice) or GDN_BF16; other values give
 *                GDN_ERR_UNSUPPORTED
 * Everything else as gdn_decode_step.
 */
GDN_API gdn_status gdn_decode_step_half_state(const gdn_problem *problem,
                                              const void *q, const void *k, const void *v,
                                              const float *g, const float *beta,
                                              void *state, int32_t state_dtype, void *out,
                                              gdn_stream_t stream);

/*
 * Verify step of speculative decoding: num_tokens (1 to 8) consecutive
 * tokens of every sequence, run from the stored state, with the output of
 * every position and the state after every position in its own slot, so
 * that the caller can keep the slot of the last accepted token.  (Page
 * "reactapp.top": the target model checks a block of draft tokens in one
 * pass and keeps the correct prefix -- section "DFlash2 : rediger sept
 * tokens en une seule passe" -- with eight speculative state slots per
 * request -- section "Pourquoi la limite est de 131 072 et non de 136 429".)
 *   problem->total_tokens == problem->num_seqs * num_tokens; token t of
 *   sequence n is row n * num_tokens + t of the token-major tensors:
 *   q, k      [N * num_tokens, Hk, dk];  v, out [N * num_tokens, Hv, dv]
 *   g, beta   [N * num_tokens, Hv] fp32
 *   state     [N, Hv, dv, dk] in state_dtype, read only
 *   slots     [N * num_tokens, Hv, dv, dk] in state_dtype: slot n *
 *             num_tokens + t = the state after token t of sequence n; must
 *             not alias state
 *   state_dtype GDN_F32, GDN_F16 or GDN_BF16; the tokens are chained in fp32
 *             registers, each slot is stored rounded (16-bit types: to
 *             nearest even)
 * Slot t equals what t + 1 successive gdn_decode_step (or
 * gdn_decode_step_half_state) calls would leave.
 */
GDN_API gdn_status gdn_verify_step(const gdn_problem *problem, int32_t num_tokens,
                                   const void *q, const void *k, const void *v,
                                   const float *g, const float *beta,
                                   const void *state, int32_t state_dtype,
                                   void *slots, void *out, gdn_stream_t stream);

/*
 * gdn_chunk_prefill without caller-provided scratch.  (The paper has no
 * counterpart: this exists for callers that cannot allocate device memory
 * when they call the layer -- engines that reserve nearly all device memory
 * for their own pools at start-up, plug-ins inside a framework that owns the
 * allocator, latency-critical paths that cannot afford cudaMalloc's
 * device-wide synchronisation.)
 *
 * Same arguments and results as gdn_chunk_prefill; problem->workspace and
 * problem->workspace_bytes are ignored.  The scratch is one 64 MiB array in
 * device memory, built into the library and held by every GPU that loads it
 * until the process exits.  Problems whose workspace size (see
 * gdn_chunk_prefill_workspace_size) exceeds 64 MiB are rejected with
 * GDN_ERR_WORKSPACE before any launch.  The first call on a device, with that
 * device current, looks up the array's device address; make that first call
 * before any stream capture.  All calls share the array: calls that may run
 * at the same time on the GPU (unordered streams) race and must be ordered by
 * the caller.  Nothing is allocated or freed.
 */
GDN_API gdn_status gdn_chunk_prefill_noalloc(const gdn_problem *problem,
                                             const void *q, const void *k, const void *v,
                                             const float *g, const float *beta,
                                             const int32_t *cu_seqlens,
                                             const float *initial_state,
                                             void *out, float *final_state,
                                             gdn_stream_t stream);

/*
 * Device-side status of the last bf16 (d = 128) prefill that ran with a given
 * workspace.  Those kernels keep an error word at the start of their
 * workspace: they cannot return a status themselves, and they do not fault
 * on the two conditions they detect.  This call waits for `stream` (it is the
 * one entry point that synchronises) and reads that word:
 *   GDN_OK             no condition recorded
 *   GDN_ERR_INVALID_ARG cu_seqlens was malformed (cu[0] != 0, decreasing, or
 *                      cu[N] != T); the prefill then wrote no output and no
 *                      final state
 *   GDN_ERR_TIMEOUT    a bounded wait inside a kernel ran out (each wait
 *                      gives up after about two seconds); outputs incomplete
 *   GDN_ERR_CUDA       the stream reports an error, or the read failed
 * Builds with GDN_DEBUG (the libgdn_debug variant) also check on the device,
 * after the call's kernels, the inputs' documented preconditions (g finite
 * and <= 0, beta in [0, 1], q and k rows of unit L2 norm within 1e-2) and
 * report a violation as GDN_ERR_INVALID_ARG (the outputs are computed all
 * the same), and they check the kernels' table-derived indices: a failure
 * is GDN_ERR_INTERNAL (a library bug; the access is skipped and the call's
 * outputs are incomplete).  The first condition recorded is the one reported.
 * workspace: problem->workspace of that gdn_chunk_prefill call, or NULL for
 * the built-in scratch of gdn_chunk_prefill_noalloc on the current device.
 * Meaningless after calls that need no workspace (fp32 inputs, d = 64).
 */
GDN_API gdn_status gdn_chunk_prefill_device_status(const void *workspace, gdn_stream_t stream);

/* Same type as cudaEvent_t. */
typedef struct CUevent_st *gdn_event_t;

/*
 * gdn_chunk_prefill with per-kernel timing, for measurement.  The call
 * records four caller-created CUDA events on `stream`: events[0] before the
 * chunk-table kernel, events[1] after it, events[2] after the prep kernel and
 * events[3] after the recurrence.  The launches are then made without
 * programmatic dependent launch, so each pair of events brackets one kernel.
 * When prep and the recurrence run as one fused launch (see
 * gdn_chunk_prefill), events[1] and events[2] mark the same point and
 * events[3] follows the fused kernel; *fused (if not NULL) is set to 1 in
 * that case (2 for the fused variant with one recurrence per value head)
 * and 0 otherwise.  With no sequences the four events are recorded
 * back to back.  Nothing is kept between calls: calls on several streams or
 * threads time themselves independently.
 *   events   four valid events (cudaEventCreate), owned by the caller;
 *            GDN_ERR_INVALID_ARG if the array or an event is NULL
 * Only for bf16 q/k/v with dk = dv = 128 (otherwise GDN_ERR_UNSUPPORTED).
 * Everything else as gdn_chunk_prefill.
 */
GDN_API gdn_status gdn_chunk_prefill_timed(const gdn_problem *problem,
                                           const void *q, const void *k, const void *v,
                                           const float *g, const float *beta,
                                           const int32_t *cu_seqlens,
                                           const float *initial_state,
                                           void *out, float *final_state,
                                           gdn_event_t const *events, int32_t *fused,
                                           gdn_stream_t stream);

/*
 * Choice of the fused prep + recurrence kernel for later prefills (process
 * wide, an atomic integer): 0 never, 1 whenever it can run, 2 when expected
 * to be faster (the default), 3 the variant with one recurrence per value
 * head whenever it can run (Hv + 16 <= SMs), even where the (sequence, value
 * head) recurrences would fit.  Any other value only queries.  Returns the
 * previous mode.
 */
GDN_API int32_t gdn_prefill_fused_mode(int32_t mode);

/*
 * Which kernels gdn_chunk_prefill would run for `problem` on a GPU with
 * `sms` SMs on which the fused kernels fit one CTA per SM (GB300: 152), in
 * fused mode `mode` (0-3 as gdn_prefill_fused_mode; any other value: the
 * current mode): 0 separate prep and recurrence kernels, 1 the fused kernel
 * with one recurrence per (sequence, value head), 2 the fused kernel with one
 * recurrence per value head over all sequences.  The choice uses only the
 * problem's sizes (total tokens and sequence count, not the lengths, which
 * are on the device).  A diagnostic: it needs no device and launches nothing.
 * Returns -1 for an invalid descriptor, a negative `sms`, or a configuration
 * without the tensor-core path (not bf16 with dk = dv = 128).
 */
GDN_API int32_t gdn_prefill_path(const gdn_problem *problem, int32_t sms, int32_t mode);

/*
 * Diagnostics for tests of the intra-chunk prep on its own (the pages compare
 * every kernel of the chunked layer with a reference separately: page
 * "cf-1.com", section "精度").  Only for bf16 q/k/v with dk = dv = 128
 * (otherwise GDN_ERR_UNSUPPORTED).
 *
 * gdn_chunk_prefill_prep_only runs the first two kernels of
 * gdn_chunk_prefill -- the chunk table and the prep -- on `stream` and leaves
 * their results in problem->workspace (argument checks and errors as
 * gdn_chunk_prefill; v, out and the states are not needed).
 *
 * gdn_chunk_prefill_prep_layout fills layout[0..7]:
 *   [0] byte offset of the slot array in the workspace; [1] bytes per slot.
 *   Slot (c, h) -- chunk c of the batch (chunks numbered sequence by
 *   sequence, 64 tokens each, the last of a sequence possibly shorter) and
 *   value head h -- starts at layout[0] + (c * Hv + h) * layout[1].  Within a
 *   slot, byte offsets of:
 *   [2] W^T = (T diag(b e^gamma) K)^T   128 rows (dk) x 64 columns (tokens)
 *   [3] T diag(b)                       64 x 64
 *   [4] P = M o Q K^T                   64 x 64
 *   [5] diag(e^gamma) Q                 two 64 x 64 images: dk 0-63, 64-127
 *   [6] e^{gamma_t}                     fp32 [64]
 *   [7] e^{gamma_L - gamma_t}           fp32 [64]
 *   (T = (I + A)^-1, A_ti = b_t e^{gamma_t - gamma_i} (k_t . k_i) for i < t,
 *   M_ri = e^{gamma_r - gamma_i} for i <= r, gamma = cumsum(g) in the chunk;
 *   tokens past a sequence's end count as b = 0, g = 0.)  The matrices are
 *   bf16 images of rows of 128 bytes (64 elements): element (r, c) is at byte
 *   128 r + 16 ((c / 8) xor (r mod 8)) + 2 (c mod 8).
 */
GDN_API gdn_status gdn_chunk_prefill_prep_only(const gdn_problem *problem,
                                               const void *q, const void *k,
                                               const float *g, const float *beta,
                                               const int32_t *cu_seqlens, gdn_stream_t stream);
GDN_API gdn_status gdn_chunk_prefill_prep_layout(const gdn_problem *problem, int64_t *layout);

/* Static, human-readable name of a status code. */
GDN_API const char *gdn_status_string(gdn_status status);

/* ABI version: major * 10000 + minor * 100 + patch. */
GDN_API int gdn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
