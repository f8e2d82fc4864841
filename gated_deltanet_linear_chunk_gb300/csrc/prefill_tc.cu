// prefill_tc.cu -- chunked prefill on the tcgen05 tensor cores (bf16 q/k/v,
// d_k = d_v = 128), as three launches on one stream:
//
//   1. gdn_chunk_table_kernel  one CTA: chunk offsets of every sequence, a
//      (sequence, first token, length) table of all chunks and the order in
//      which the recurrence CTAs take sequences (longest first).
//   2. gdn_prep_kernel         one unit of 128 threads per (chunk, value
//      head) item, all chunks at once: the intra-chunk prep,
//        gamma = cumsum(g); [K; Q] K^T in one M = 128 MMA (K K^T and Q K^T);
//        A_ti = b_t e^{gamma_t - gamma_i} (k_t . k_i), i < t;
//        T = (I + A)^-1 as  T = D' - (D' E) D',  where D' holds the inverses
//          of the two 32 x 32 diagonal blocks of I + A (each from its two
//          16 x 16 diagonal blocks, inverted by fp32 forward substitution
//          and merged by two MMAs) and E the lower-left block of A (two
//          MMAs; with only two blocks, (D' E)^2 = 0, so the series stops
//          there);
//        W^T = K^T (T diag(b e^gamma))^T  (MMA, M = 128);
//        P = M o Q K^T,  M_ri = e^{gamma_r - gamma_i} for i <= r;
//      and stores W^T, T diag(b), P, diag(e^gamma) Q (bf16, as swizzled
//      shared-memory tile images), e^gamma and e^{gamma_L - gamma} in the
//      workspace.
//   3. gdn_chain_kernel        one CTA per (sequence, value head): the
//      inter-chunk recurrence and the output, warp-specialised: one thread
//      issues TMA loads, one issues MMAs, eight warps run the state
//      epilogues and four the output.  The fp32 state S (dv x dk) stays in
//      tensor memory for the whole sequence (as sigma S^, a running scale
//      times a stored state); per chunk, with a bf16 copy -S0 of the chunk's
//      start state in tensor memory as the MMA operand:
//         Delta^T = V^T (T diag b)^T - S0 W^T       (both MMAs into one tile)
//         S      <- e^{gamma_L} S + (diag(e^{gamma_L - gamma}) Delta)^T K
//         O^T     = diag(e^gamma)-scaled S0 Q^T + Delta^T P^T
//      The two MMAs that carry the state from chunk to chunk (S0 W^T, then
//      the update of S) and their epilogues are the critical path; the output
//      MMAs and the next chunk's loads run beside them.
//
// Instead of 2 and 3, gdn_fused_kernel can run both in one cooperative
// launch: the recurrences on some SMs, the prep units on the others, each
// recurrence waiting for a ready flag per (chunk, value head) before it loads
// the chunk.
//
// The algorithm is the chunked (WY/UT) form of the Gated DeltaNet recurrence
// with chunk length 64, split into intra-chunk prep, inter-chunk state
// recurrence and output, as the page "cf-1.com" (section "三个优化", item 2
// "GDN prefill") describes its three kernels; that page keeps the state in
// mma accumulator registers on Turing, here it lives in Blackwell tensor
// memory and the next chunk's inputs arrive by TMA while the current one is
// used.
//
// Tokens past the end of a sequence inside its last chunk get b = 0 and
// g = 0, which zeroes their rows of W, U and Delta and keeps gamma_L at the
// last real token.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "sm103.cuh"

namespace gdn {
namespace {

using namespace ptx;

constexpr int C = 64;           // chunk length
constexpr int D = 128;          // head dim (dk = dv)
constexpr int kTile = 8192;     // bytes of one 64 x 64 bf16 swizzled tile
constexpr int kMaxSortSeqs = 4096;
constexpr float kLog2e = 1.4426950408889634f;


// Per (chunk, value head) slot written by the prep kernel.
constexpr int kSlotWT = 0;                    // W^T  [128 dk][64 tokens], MN-major B image
constexpr int kSlotTB = kSlotWT + 2 * kTile;  // T diag(b) [64 out][64 in], K-major B image
constexpr int kSlotP = kSlotTB + kTile;       // P [64 out][64 in], K-major B image
constexpr int kSlotQ = kSlotP + kTile;        // diag(e^gamma) Q [64 tokens][128 dk], K-major B image
constexpr int kSlotEG = kSlotQ + 2 * kTile;   // e^{gamma_t}, fp32 [64]
constexpr int kSlotDEC = kSlotEG + 256;       // e^{gamma_L - gamma_t}, fp32 [64]
constexpr int kSlotBytes = kSlotDEC + 256;    // 49664

// ------------------------------------------------------------------ workspace
struct WsLayout {
    size_t hdr, chunk_off, snap_off, order, table, gl, tiles, flags, porder, total;
    int64_t max_chunks;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

WsLayout ws_layout(const gdn_problem &p) {
    WsLayout w;
    w.max_chunks = (p.total_tokens + C - 1) / C + p.num_seqs;
    w.hdr = 0;
    w.chunk_off = 256;
    w.snap_off = align_up(w.chunk_off + 4 * (size_t)(p.num_seqs + 1), 256);
    w.order = align_up(w.snap_off + 4 * (size_t)(p.num_seqs + 1), 256);
    w.table = align_up(w.order + 4 * (size_t)p.num_seqs, 256);
    w.gl = align_up(w.table + 16 * (size_t)w.max_chunks, 256);  // e^{gamma_L} per (chunk, value head)
    w.tiles = align_up(w.gl + 4 * (size_t)w.max_chunks * p.num_v_heads, 1024);
    // Ready flag per (chunk, value head) for the fused prep + recurrence kernel,
    // then the ticket its prep units draw items from,
    w.flags = w.tiles + (size_t)w.max_chunks * p.num_v_heads * kSlotBytes;
    // and the order in which its prep units take the chunks.
    w.porder = align_up(w.flags + 4 * ((size_t)w.max_chunks * p.num_v_heads + 1), 256);
    w.total = align_up(w.porder + 4 * (size_t)w.max_chunks, 256);
    return w;
}

// ------------------------------------------------------------------ kernel 1
// One CTA of 1024 threads.  chunk_off[n] = number of chunks before sequence n
// (chunk_off[N] = total), table[chunk] = {n, first token, length, index in
// sequence}, order = sequences by decreasing chunk count (stable), identity
// when N is large.  Malformed cu_seqlens (not starting at 0, decreasing, not
// ending at T, or more chunks than the workspace holds) record an error and
// make the whole call a no-op.
// Sequences whose chunk offsets the table kernel keeps in shared memory
// (more than this: it reads them back from the workspace).
constexpr int kTableSmemSeqs = 4096;

// Inclusive sum over the warp of x (lane order).
__device__ __forceinline__ int warp_incl_scan(int x) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    return x;
}

__global__ void __launch_bounds__(1024)
gdn_chunk_table_kernel(const int32_t *__restrict__ cu, int N, int64_t T, int64_t max_chunks,
                       int snap_stride, int *__restrict__ err, int *__restrict__ chunk_off,
                       int *__restrict__ snap_off, int *__restrict__ order,
                       int4 *__restrict__ table, unsigned *__restrict__ flags, int n_flags,
                       int *__restrict__ porder) {
    __shared__ int s_off[kTableSmemSeqs + 1];
    __shared__ int s_wsum[32], s_wsum2[32];
    __shared__ int s_carry, s_carry2;
    __shared__ int s_bad;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool in_smem = N <= kTableSmemSeqs;
    griddep_launch_dependents();  // prep may be scheduled; it waits for this grid
    for (int i = tid; i < n_flags; i += 1024) flags[i] = 0u;
    if (tid == 0) {
        s_carry = 0;
        s_carry2 = 0;
        s_bad = (cu[0] != 0 || (int64_t)cu[N] != T) ? 1 : 0;
        *err = kErrNone;
    }
    __syncthreads();
    // Chunk (and snapshot slot) offsets: a scan over the sequences, 1024 at a
    // time (warp scans, then a scan of the 32 warp sums).
    for (int base = 0; base < N; base += 1024) {
        const int n = base + tid;
        int nch = 0;
        if (n < N) {
            const int len = cu[n + 1] - cu[n];
            if (len < 0) s_bad = 1;
            nch = len > 0 ? (len + C - 1) / C : 0;
        }
        // Snapshot slots of the sequence: one per snap_stride chunks, the
        // last chunk always included.
        const int nsn = (n < N && snap_stride > 0) ? (nch + snap_stride - 1) / snap_stride : 0;
        const int a = warp_incl_scan(nch), a2 = warp_incl_scan(nsn);
        if (lane == 31) {
            s_wsum[warp] = a;
            s_wsum2[warp] = a2;
        }
        __syncthreads();
        if (warp == 0) {
            s_wsum[lane] = warp_incl_scan(s_wsum[lane]);
            s_wsum2[lane] = warp_incl_scan(s_wsum2[lane]);
        }
        __syncthreads();
        const int pre = s_carry + (warp > 0 ? s_wsum[warp - 1] : 0);
        const int pre2 = s_carry2 + (warp > 0 ? s_wsum2[warp - 1] : 0);
        if (n < N) {
            chunk_off[n] = pre + a - nch;
            snap_off[n] = pre2 + a2 - nsn;
            if (in_smem) s_off[n] = pre + a - nch;
        }
        __syncthreads();
        if (tid == 0) {
            s_carry += s_wsum[31];
            s_carry2 += s_wsum2[31];
        }
        __syncthreads();
    }
    if (tid == 0) {
        if ((int64_t)s_carry > max_chunks) s_bad = 1;
        if (s_bad) *err = kErrCuSeqlens;
        snap_off[N] = s_carry2;
        chunk_off[N] = s_bad ? 0 : s_carry;
        if (in_smem) s_off[N] = s_carry;
    }
    __syncthreads();
    if (s_bad) {
        for (int n = tid; n < N; n += 1024) chunk_off[n] = 0;
        if (order)
            for (int n = tid; n < N; n += 1024) order[n] = n;
        return;
    }
    // Chunk offsets of this call (block-visible: shared memory, or the
    // workspace written above).
    const int *off = in_smem ? s_off : chunk_off;
    const int total = s_carry;
    for (int ch = tid; ch < total; ch += 1024) {
        int lo = 0, hi = N - 1;  // last n with off[n] <= ch
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (off[mid] <= ch) lo = mid; else hi = mid - 1;
        }
        const int c = ch - off[lo];
        const int tok0 = cu[lo] + c * C;
        table[ch] = make_int4(lo, tok0, min(C, cu[lo + 1] - tok0), c);
        if (porder) {
            // Rank of the chunk by (position in its sequence, sequence): the
            // fused kernel's prep takes every sequence's chunk c before any
            // chunk c + 1.
            int rank = 0;
            for (int m = 0; m < N; ++m) {
                const int nm = off[m + 1] - off[m];
                rank += min(c, nm) + ((m < lo && nm > c) ? 1 : 0);
            }
            porder[rank] = ch;
        }
    }
    for (int n = tid; order && n < N; n += 1024) {
        if (N > kMaxSortSeqs) {
            order[n] = n;
            continue;
        }
        const int mine = off[n + 1] - off[n];
        int rank = 0;
        for (int m = 0; m < N; ++m) {
            const int other = off[m + 1] - off[m];
            rank += (other > mine) || (other == mine && m < n);
        }
        order[rank] = n;
    }
}


// Inclusive prefix sum of g over one chunk (lane holds tokens 2l, 2l+1),
// with g = 0 past the end of the sequence.  Optionally also b (0 past the
// end), e^{gamma_t}, e^{gamma_L - gamma_t} and e^{-gamma_t}.  Called by one
// full warp.
// The arithmetic of chunk_gamma on the lane's tokens' g (and b) values.
__device__ __forceinline__ void chunk_gamma_of(float g0, float g1, float b0, float b1, float *gam,
                                               float *beta_out, float *eg, float *dec,
                                               float *einv) {
    const int lane = threadIdx.x & 31;
    const int t0 = 2 * lane, t1 = 2 * lane + 1;
    float s = g0 + g1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float x = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += x;
    }
    const float ga = s - g1, gb = s;
    gam[t0] = ga;
    gam[t1] = gb;
    beta_out[t0] = b0;
    beta_out[t1] = b1;
    const float gL = __shfl_sync(0xffffffffu, s, 31);
    eg[t0] = expf(ga);
    eg[t1] = expf(gb);
    dec[t0] = expf(gL - ga);
    dec[t1] = expf(gL - gb);
    einv[t0] = expf(-ga);
    einv[t1] = expf(-gb);
}

__device__ __forceinline__ void chunk_gamma(const float *__restrict__ g, int tok0, int L, int Hv,
                                            int h, float *gam, float *beta_out,
                                            const float *__restrict__ beta, float *eg = nullptr,
                                            float *dec = nullptr, float *einv = nullptr) {
    const int lane = threadIdx.x & 31;
    const int t0 = 2 * lane, t1 = 2 * lane + 1;
    const float g0 = t0 < L ? g[(size_t)(tok0 + t0) * Hv + h] : 0.f;
    const float g1 = t1 < L ? g[(size_t)(tok0 + t1) * Hv + h] : 0.f;
    if (beta_out && eg && einv) {
        const float b0 = t0 < L ? beta[(size_t)(tok0 + t0) * Hv + h] : 0.f;
        const float b1 = t1 < L ? beta[(size_t)(tok0 + t1) * Hv + h] : 0.f;
        chunk_gamma_of(g0, g1, b0, b1, gam, beta_out, eg, dec, einv);
        return;
    }
    float s = g0 + g1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float x = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += x;
    }
    const float ga = s - g1, gb = s;
    gam[t0] = ga;
    gam[t1] = gb;
    if (beta_out) {
        beta_out[t0] = t0 < L ? beta[(size_t)(tok0 + t0) * Hv + h] : 0.f;
        beta_out[t1] = t1 < L ? beta[(size_t)(tok0 + t1) * Hv + h] : 0.f;
    }
    if (eg) {
        const float gL = __shfl_sync(0xffffffffu, s, 31);
        eg[t0] = expf(ga);
        eg[t1] = expf(gb);
        dec[t0] = expf(gL - ga);
        dec[t1] = expf(gL - gb);
    }
    if (einv) {
        einv[t0] = expf(-ga);
        einv[t1] = expf(-gb);
    }
}

// ------------------------------------------------------------------ kernel 2
// Intra-chunk prep, one (chunk, value head) item per unit of 128 threads
// (four warps, one per TMEM lane quadrant).  Small units keep many items in
// flight on an SM (four per CTA of the fused kernel, five CTAs per SM of the
// separate kernel): an item is a chain of dependent steps (tile loads, six
// MMA round trips, CUDA-core epilogues between barriers), and independent
// items fill each other's waits.  Within an item one warp polls each
// mbarrier while the others block at the unit's named barrier (no issue
// slots spent waiting), TMEM rows are read eight columns at a time in rolled
// loops (little code for the instruction cache), and the slot's large
// images leave through shared memory by bulk copies.  The K K^T and Q K^T
// product is recomputed for each value head of a key head; it is one small
// MMA.
constexpr int kPrepThreads = 128;
constexpr int kPrepUnits = 4;              // units per CTA of the fused kernel
constexpr int kPrepCtasPerSm = 5;          // one-unit CTAs per SM of the separate kernel
constexpr uint32_t kPrepTmemCols = 64;     // [K; Q] K^T, then N, Y and W^T in turn
// Below this gamma_L the factors e^{gamma_t} and e^{-gamma_i} of A and P could
// overflow fp32 (e^{-gamma_i} <= e^{-gamma_L}): such chunks take one
// exponential per element instead.
constexpr float kFactorGammaMin = -80.f;
// The unit's thread that issues its TMA loads and bulk copies and publishes
// its items (thread 0 issues the MMAs and its warp polls the mbarriers).
constexpr int kCopier = 96;

struct alignas(1024) PrepSmem {
    // K atom 0 | Q atom 0 | K atom 1 | Q atom 1 (two 64-column 128-byte-swizzled
    // atoms each, stacked so that one M = 128 MMA gives K K^T and Q K^T).  The
    // Q atoms are scaled in place to diag(e^gamma) Q and copied to the slot;
    // then Q atom 0 holds A16 (A below its diagonal 16 x 16 blocks, bf16),
    // which becomes E, then N = D' E; Q atom 1 holds XD (the inverses of the
    // diagonal 16 x 16 blocks of I + A, bf16), which becomes D', then
    // T diag(b) (copied to the slot).  K atom 0 + Q atom 0 finally stage W^T
    // (copied to the slot).
    uint8_t kq[4 * kTile];
    // A's four diagonal 16 x 16 blocks (fp32) for the forward substitution;
    // then T diag(b e^gamma) (bf16, the W^T MMA's operand).
    uint8_t ab[kTile];
    float gam[C];
    float beta[C];
    float eg[C];    // e^{gamma_t}
    float einv[C];  // e^{-gamma_t}
    float dec[C];   // e^{gamma_L - gamma_t}
    float bg[C];    // b_t e^{gamma_t}
    int4 nxt[2];    // chunk-table entries of this and the next item: {chunk, head, token, length}
    uint64_t tma_bar;
    uint64_t mma_bar;
    uint32_t tmem;
    int fact;       // the chunk's A and P factorise (gamma_L >= kFactorGammaMin)
};

// Row r of A's fp32 diagonal 16 x 16 block b in ab: 16 floats; blocks 260
// floats apart (so that rows of two blocks read at once fall in different
// banks).
__device__ __forceinline__ float *adiag(PrepSmem &sm, int b, int r) {
    return reinterpret_cast<float *>(sm.ab) + 260 * b + 16 * r;
}

// Element (r, c) of a bf16 image with 128-byte swizzled rows.
__device__ __forceinline__ __nv_bfloat16 *img_at(uint8_t *img, int r, int c) {
    return reinterpret_cast<__nv_bfloat16 *>(img + swz(r, c >> 3) + 2 * (c & 7));
}

// Writes 8 floats as one 16-byte bf16 chunk.
__device__ __forceinline__ uint4 pack8(const float *x) {
    return make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]),
                      pack_bf16(x[6], x[7]));
}

__device__ __forceinline__ void unpack8(uint4 w, float *x) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162 *>(&u[k]);
        const float2 f = __bfloat1622float2(b2);
        x[2 * k] = f.x;
        x[2 * k + 1] = f.y;
    }
}

__device__ __forceinline__ void tmem_ld32f(uint32_t taddr, float (&x)[32]) {
    uint32_t r[32];
    tmem_ld32(taddr, r);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(r[i]);
}

// Eight elements s e^{gamma_r - gamma_i} x_i of a row r of A (with b_r in s)
// or P, columns i0 .. i0 + 7 read from TMEM; entries past `last` are 0.
// kFact: e^{gamma_r - gamma_i} = e^{gamma_r} e^{-gamma_i} (rs = s e^{gamma_r});
// else one exponential per element.
template <bool kFact>
__device__ __forceinline__ void decayed8(const PrepSmem &sm, uint32_t taddr, int i0, int last,
                                         float s, float rs, float gr, float (&a)[8]) {
    uint32_t r[8];
    tmem_ld8(taddr, r);
    const float4 *src4 = reinterpret_cast<const float4 *>(kFact ? sm.einv + i0 : sm.gam + i0);
    const float4 f0 = src4[0], f1 = src4[1];
    const float f[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
    tmem_ld_wait();
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const float x = __uint_as_float(r[u]);
        const float v = kFact ? rs * f[u] * x : s * ex2_approx((gr - f[u]) * kLog2e) * x;
        a[u] = i0 + u <= last ? v : 0.f;
    }
}

// decayed8 with the factorised form chosen once for the chunk (a branch
// that is the same for the whole unit, outside the loops).
#define DECAYED8(taddr, i0, last, s, rs, gr, a)                        \
    do {                                                                \
        if (fact) decayed8<true>(sm, taddr, i0, last, s, rs, gr, a);   \
        else decayed8<false>(sm, taddr, i0, last, s, rs, gr, a);       \
    } while (0)

// The unit's wait for an mbarrier phase: warp 0 polls (bounded), then the
// whole unit meets at its named barrier, which also ORs the failure flags.
// True when the unit must stop.
__device__ __forceinline__ bool unit_wait(uint64_t *bar, uint32_t parity, int warp, int nbar,
                                          bool bad) {
    if (warp == 0 && !bad) bad = !warp_wait_poll(bar, parity);
    return named_barrier_or(nbar, kPrepThreads, bad);
}

// Makes an item's slot visible device-wide and publishes its ready flag
// (the thread that issued the slot's bulk copies, all of them this thread's
// committed groups; every other thread's slot writes are ordered before a
// unit barrier this thread has passed since).  The copies are complete and
// ordered before the flag by the proxy fence; the release store at device
// scope carries them, and, through the barrier, the other threads' writes, to
// a reader that acquires the flag (no further fence is needed).
__device__ __forceinline__ void publish_item(unsigned *flag, unsigned epoch) {
    bulk_wait_group<0>();
    fence_proxy_async_global();
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(flag), "r"(epoch) : "memory");
}

// One prep unit: kPrepThreads threads with local index `ltid` (the unit's
// first warp is a multiple of 4, so warp w of the unit reads TMEM lane
// quadrant w), its own PrepSmem, TMEM columns and named barriers `bar` (the
// unit) and `bar2` (its warps 2 and 3).  Items are numbered chunk * Hv +
// value head (chunk-major, chunks in the prep order when `porder` is given),
// below n_items.  With `flags`, each finished item publishes `epoch` into
// flags[chunk * Hv + h] (release, device scope) once its workspace slot is
// written.  kLoop = false: exactly the one item item0, compiled without the
// loop.
// `relinquish`: give up the CTA's TMEM allocation permit after allocating
// (only when the CTA allocates nothing after this unit).  kLoop units also
// take `ticket`: their first two items are item0 and item0 + stride (the
// grid's first two rounds, in order), the later ones are drawn one at a time
// from *ticket (item = dyn0 + ticket, in order, while items remain), so that
// a unit slowed down holds up only the item it is on.  The next item is drawn
// during the current one (the ticket, the prep order and the chunk table read
// a few phases apart) into the unit's two-entry ring `nxt`.  Every item's
// flag is published as soon as its slot is written.  (A look-ahead that
// loaded each item's tiles, g and beta during the item before, and deferred
// each flag to the next item, was slower: the first pass of its larger code
// through an SM cost more than it saved.)
//
// Per item:
//   gamma = cumsum(g), b, e^gamma, e^{gamma_L - gamma};  [K; Q] K^T (M = 128);
//   diag(e^gamma) Q to the slot;
//   A_ti = b_t e^{gamma_t - gamma_i} (k_t . k_i), i < t: its diagonal 16 x 16
//     blocks in fp32, the rest below them (E included) in bf16;
//   P = M o Q K^T, M_ri = e^{gamma_r - gamma_i} (i <= r), to the slot;
//   D' = blockdiag((I + A_bb)^-1), each 32 x 32 block from its two 16 x 16
//     diagonal blocks (fp32 forward substitution) and the merge
//     [[X1, 0], [-X2 C X1, X2]] (C the lower-left 16 x 16 block; two M = 64
//     MMAs);
//   T = (I + A)^-1 = D' - (D' E) D' (two M = 64 MMAs: with two blocks
//     (D' E)^2 = 0, so the series stops there);
//   T diag(b) to the slot, W^T = K^T (T diag(b e^gamma))^T (M = 128) to the slot.
template <bool kLoop>
__device__ __forceinline__ void prep_unit(
    PrepSmem &sm, const CUtensorMap *tm_q, const CUtensorMap *tm_k, const float *__restrict__ g,
    const float *__restrict__ beta, const int *__restrict__ chunk_off,
    const int4 *__restrict__ table, uint8_t *__restrict__ slots, float *__restrict__ gl,
    int *__restrict__ err, int N, int Hk, int Hv, int ltid, int bar, int bar2, int item0,
    int stride, int n_items, unsigned *flags, unsigned epoch, bool relinquish,
    const int *__restrict__ porder = nullptr, unsigned *ticket = nullptr, int dyn0 = 0) {
    const int tid = ltid, warp = tid >> 5, lane = tid & 31;
    const int G = Hv / Hk;
    const int q4 = (threadIdx.x >> 5) & 3;  // TMEM lane quadrant of the physical warp
    const int row = 32 * q4 + lane;         // this thread's TMEM lane
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
    uint8_t *const bufE = sm.kq + kTile;      // Q atom 0
    uint8_t *const bufD = sm.kq + 3 * kTile;  // Q atom 1
    const int n_ch = chunk_off[N];
    auto chunk_of = [&](int item) { return item / Hv; };
    // Chunk-table entry of an item: {chunk, value head, first token, length}.
    auto locate = [&](int item) {
        const int ci = chunk_of(item);
        const int ch = porder ? porder[ci] : ci;
        const int4 e = table[ch];
        return make_int4(ch, item % Hv, e.y, e.z);
    };

    if (tid == 0) {
        prefetch_tensormap(tm_q);
        prefetch_tensormap(tm_k);
        mbar_init(&sm.tma_bar, 1);
        mbar_init(&sm.mma_bar, 1);
        fence_mbar_init();
        // The first item's entry (chunk -1 when there is none).
        sm.nxt[0] = (item0 < n_items && chunk_of(item0) < n_ch) ? locate(item0)
                                                                 : make_int4(-1, 0, 0, 0);
    }
    if (warp == 0) {
        tmem_alloc(&sm.tmem, kPrepTmemCols);
        // The permit is the CTA's: with several units in one CTA (kLoop) the
        // others may still have to allocate.
        if (relinquish) tmem_relinquish();
    }
    tc_fence_before();
    named_barrier(bar, kPrepThreads);
    tc_fence_after();
    const uint32_t tmem = sm.tmem;
    bool bad = false;
    uint32_t mph = 0, tph = 0;
    int it = 0;
#pragma unroll 1
    for (; !bad; ++it) {
        if (sm.nxt[it & 1].x < 0) break;
        const int4 cur = sm.nxt[it & 1];
        const int ch = cur.x, h = cur.y, tok0 = cur.z, L = cur.w, hk = h / G;
        if (kDebug && !(ch >= 0 && ch < n_ch && h >= 0 && h < Hv && tok0 >= 0 && L >= 1 && L <= C)) {
            if (tid == 0) debug_fail(err, kErrIndex);  // (then the unit stops, as on a time-out)
            bad = true;
            break;
        }
        uint8_t *const slot = slots + ((size_t)ch * Hv + h) * kSlotBytes;
        // (kLoop: warp 2, lane 0) the next item: its number, whether it
        // exists, its chunk from the prep order and its chunk-table entry
        int item2 = 0, pch = 0;
        bool more2 = false;
        if (tid == kCopier) {
            if (kLoop) {
                // The previous item's bulk copies have read the tiles, and
                // its generic accesses are ordered before the TMA writes.
                bulk_wait_group_read<0>();
                fence_proxy_async_smem();
            }
            mbar_arrive_expect_tx(&sm.tma_bar, 4 * kTile);
            tma_load_3d(sm.kq + 0 * kTile, tm_k, 0, hk, tok0, &sm.tma_bar);
            tma_load_3d(sm.kq + 1 * kTile, tm_q, 0, hk, tok0, &sm.tma_bar);
            tma_load_3d(sm.kq + 2 * kTile, tm_k, 64, hk, tok0, &sm.tma_bar);
            tma_load_3d(sm.kq + 3 * kTile, tm_q, 64, hk, tok0, &sm.tma_bar);
        }
        if (warp == 1) {
            // gamma, b and the decay factors while the tiles are in flight
            chunk_gamma(g, tok0, L, Hv, h, sm.gam, sm.beta, beta, sm.eg, sm.dec, sm.einv);
            float *slot_f = reinterpret_cast<float *>(slot);
            slot_f[kSlotEG / 4 + 2 * lane] = sm.eg[2 * lane];
            slot_f[kSlotEG / 4 + 2 * lane + 1] = sm.eg[2 * lane + 1];
            slot_f[kSlotDEC / 4 + 2 * lane] = sm.dec[2 * lane];
            slot_f[kSlotDEC / 4 + 2 * lane + 1] = sm.dec[2 * lane + 1];
            sm.bg[2 * lane] = sm.beta[2 * lane] * sm.eg[2 * lane];
            sm.bg[2 * lane + 1] = sm.beta[2 * lane + 1] * sm.eg[2 * lane + 1];
            if (lane == 31) {
                gl[(size_t)ch * Hv + h] = sm.eg[C - 1];
                sm.fact = sm.gam[C - 1] >= kFactorGammaMin;
            }
        } else if (kLoop && warp == 2 && lane == 0) {
            // The next item: the second static round, then the ticket (its
            // value first read after the unit barrier below).
            item2 = it == 0 ? item0 + stride : dyn0 + (int)atomicAdd(ticket, 1u);
        }
        if ((bad = unit_wait(&sm.tma_bar, tph, warp, bar, bad))) break;
        tph ^= 1;
        if (kLoop && warp == 2 && lane == 0) {
            more2 = item2 < n_items && chunk_of(item2) < n_ch;
            if (more2) pch = porder ? porder[chunk_of(item2)] : chunk_of(item2);
        }
        if (tid == 0) {
            tc_fence_after();
            const uint32_t base = smem_u32(sm.kq);
            constexpr uint32_t id = idesc_bf16(128, 64, false, false);
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
                const uint32_t off = (k / 4) * (2 * kTile) + (k % 4) * 32;
                mma_bf16(tmem, smem_desc(base + off, 16, 1024), smem_desc(base + off, 16, 1024),
                         id, k > 0);
            }
            mma_commit(&sm.mma_bar);
        }
        if ((bad = unit_wait(&sm.mma_bar, mph, warp, bar, bad))) break;
        mph ^= 1;
        tc_fence_after();
        // ---- diag(e^gamma) Q in place in the Q atoms, then copied to the slot.
        // A thread scales 16-byte chunk tid % 8 of rows tid / 8 + 16 j of both
        // atoms (rows 16 apart share the swizzle, so the address steps by 2 KB).
        {
            const int r0 = tid >> 3;
            uint8_t *p0 = sm.kq + kTile + swz(r0, tid & 7);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                uint4 *p = reinterpret_cast<uint4 *>(p0 + (j >> 2) * (2 * kTile) + (j & 3) * 2048);
                const float e = sm.eg[r0 + 16 * (j & 3)];
                float v[8];
                unpack8(*p, v);
#pragma unroll
                for (int u = 0; u < 8; u += 2) {
                    const float2 w = mul2(make_float2(v[u], v[u + 1]), make_float2(e, e));
                    v[u] = w.x;
                    v[u + 1] = w.y;
                }
                *p = pack8(v);
            }
        }
        fence_proxy_async_smem();
        named_barrier(bar, kPrepThreads);
        if (tid == kCopier) {
            bulk_store(slot + kSlotQ, sm.kq + kTile, kTile);
            bulk_store(slot + kSlotQ + kTile, sm.kq + 3 * kTile, kTile);
            bulk_commit_group();
        }
        // ---- A's four diagonal 16 x 16 blocks (fp32, into ab) from K K^T
        // (lanes 0-63), P from Q K^T (lanes 64-127, to the slot).  A warp's
        // TMEM loads take the same columns for every lane (warp-uniform); a
        // lane keeps the 16 of its own block.
        const bool fact = sm.fact;
        if (q4 < 2) {
            const int t = row;
            const float gt = sm.gam[t], bt = sm.beta[t], rs = bt * sm.eg[t];
#pragma unroll 1
            for (int c8 = 0; c8 < 4; ++c8) {
                float a[8];
                DECAYED8(tmem + lane_base + 32 * q4 + 8 * c8, 32 * q4 + 8 * c8, t - 1, bt, rs, gt, a);
                if ((c8 >> 1) == (lane >> 4)) {
                    float *dst = adiag(sm, t >> 4, t & 15) + 8 * (c8 & 1);
                    *reinterpret_cast<float4 *>(dst) = make_float4(a[0], a[1], a[2], a[3]);
                    *reinterpret_cast<float4 *>(dst + 4) = make_float4(a[4], a[5], a[6], a[7]);
                }
            }
        } else {
            const int r = row - 64;
            const float gr = sm.gam[r], rs = sm.eg[r];
#pragma unroll 1
            for (int c8 = 0; c8 < 8; ++c8) {
                float a[8];
                if (c8 < 4 || q4 == 3) {  // (rows 0-31 have nothing at columns 32-63)
                    DECAYED8(tmem + lane_base + 8 * c8, 8 * c8, r, 1.f, rs, gr, a);
                } else {
#pragma unroll
                    for (int u = 0; u < 8; ++u) a[u] = 0.f;
                }
                *reinterpret_cast<uint4 *>(slot + kSlotP + swz(r, c8)) = pack8(a);
            }
        }
        if (tid == kCopier) bulk_wait_group_read<0>();  // the Q atoms are free
        named_barrier(bar, kPrepThreads);
        // ---- Warps 2-3 invert the four 16 x 16 diagonal blocks of I + A by
        // forward substitution (one column per thread) into XD, the bf16
        // image in Q atom 1 that becomes D'.  Meanwhile warps 0-1 write A16,
        // the part of A below the diagonal 16 x 16 blocks (bf16, Q atom 0),
        // and clear XD outside its blocks.
        if (q4 >= 2) {
            const int ft = tid - 64, fb = ft >> 4, fcol = ft & 15;  // 16-block, column
            float xc[16];
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                float a0 = (t == fcol) ? 1.f : 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
                const float *ar = adiag(sm, fb, t);
#pragma unroll
                for (int i = 0; i < (t & ~3); i += 4) {
                    const float4 av = *reinterpret_cast<const float4 *>(ar + i);
                    a0 = fmaf(-av.x, xc[i], a0);
                    a1 = fmaf(-av.y, xc[i + 1], a1);
                    a2 = fmaf(-av.z, xc[i + 2], a2);
                    a3 = fmaf(-av.w, xc[i + 3], a3);
                }
#pragma unroll
                for (int i = (t & ~3); i < t; ++i) a0 = fmaf(-ar[i], xc[i], a0);
                xc[t] = (a0 + a1) + (a2 + a3);
                *img_at(bufD, 16 * fb + t, 16 * fb + fcol) = __float2bfloat16_rn(xc[t]);
            }
        } else {
            const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
            const int t = row, tb = t >> 4;  // (tb: the row's diagonal block)
            const float gt = sm.gam[t], bt = sm.beta[t], rs = bt * sm.eg[t];
            // A16 row t: A at columns below 16 tb, 0 from there on.  The
            // warp loads the columns its last lane needs (2 or 6 chunks).
#pragma unroll 1
            for (int c8 = 0; c8 < 8; ++c8) {
                float a[8];
                if (c8 < 2 + 4 * q4) {
                    DECAYED8(tmem + lane_base + 8 * c8, 8 * c8, t - 1, bt, rs, gt, a);
                    *reinterpret_cast<uint4 *>(bufE + swz(t, c8)) = c8 < 2 * tb ? pack8(a) : z4;
                } else {
                    *reinterpret_cast<uint4 *>(bufE + swz(t, c8)) = z4;
                }
            }
            // XD row t: zero outside chunks 2 tb, 2 tb + 1.
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8)
                if ((c8 >> 1) != tb) *reinterpret_cast<uint4 *>(bufD + swz(t, c8)) = z4;
        }
        fence_proxy_async_smem();
        tc_fence_before();  // this item's last reads of [K K^T; Q K^T]
        named_barrier(bar, kPrepThreads);
        // ---- The 16 -> 32 merge on the tensor pipe.  Y = A16 XD: in its rows
        // 16-31 x columns 0-15 and 48-63 x columns 32-47 it is C X1 of each
        // 32 x 32 diagonal block (C = its lower-left 16 x 16 block of A); the
        // rest of Y (from A's lower-left 32 x 32 block) is not used.
        if (kLoop && warp == 2 && lane == 0) {  // (the next item's entry, read at its start)
            const int4 e2 = more2 ? table[pch] : make_int4(0, 0, 0, 0);
            sm.nxt[(it + 1) & 1] = more2 ? make_int4(pch, item2 % Hv, e2.y, e2.z)
                                         : make_int4(-1, 0, 0, 0);
        }
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id = idesc_bf16(64, 64, false, true);
            const uint32_t a = smem_u32(bufE), b = smem_u32(bufD);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_bf16(tmem, smem_desc(a + 32 * k, 16, 1024), smem_desc(b + 2048 * k, kTile, 1024),
                         id, k > 0);
            mma_commit(&sm.mma_bar);
        }
        if ((bad = unit_wait(&sm.mma_bar, mph, warp, bar, bad))) break;
        mph ^= 1;
        tc_fence_after();
        // Those two 16 x 16 blocks of Y replace C in A16 (M = 64 layout: row
        // 16 q + lane in lane 32 q + lane; quadrants 1 and 3 hold them).
        const int mcol = (q4 & 2) ? 32 : 0;
        if (q4 & 1) {
            uint32_t r0[8], r1[8];
            tmem_ld8(tmem + lane_base + mcol, r0);
            tmem_ld8(tmem + lane_base + mcol + 8, r1);
            tmem_ld_wait();
            if (lane < 16) {
                const int r = 16 * q4 + lane;
                float y[16];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    y[u] = __uint_as_float(r0[u]);
                    y[8 + u] = __uint_as_float(r1[u]);
                }
                *reinterpret_cast<uint4 *>(bufE + swz(r, mcol >> 3)) = pack8(y);
                *reinterpret_cast<uint4 *>(bufE + swz(r, (mcol >> 3) + 1)) = pack8(y + 8);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        named_barrier(bar, kPrepThreads);
        // -XD Y: in the same two blocks, -X2 C X1, the lower-left 16 x 16
        // block of each 32 x 32 block of D' (A negated by the descriptor).
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id = idesc_bf16(64, 64, false, true, true);
            const uint32_t a = smem_u32(bufD), b = smem_u32(bufE);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_bf16(tmem, smem_desc(a + 32 * k, 16, 1024), smem_desc(b + 2048 * k, kTile, 1024),
                         id, k > 0);
            mma_commit(&sm.mma_bar);
        }
        if ((bad = unit_wait(&sm.mma_bar, mph, warp, bar, bad))) break;
        mph ^= 1;
        tc_fence_after();
        // Into XD (which becomes D'), and zeros back into A16 (which becomes
        // E, A's lower-left 32 x 32 block).
        if (q4 & 1) {
            uint32_t r0[8], r1[8];
            tmem_ld8(tmem + lane_base + mcol, r0);
            tmem_ld8(tmem + lane_base + mcol + 8, r1);
            tmem_ld_wait();
            if (lane < 16) {
                const int r = 16 * q4 + lane;
                float m[16];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    m[u] = __uint_as_float(r0[u]);
                    m[8 + u] = __uint_as_float(r1[u]);
                }
                *reinterpret_cast<uint4 *>(bufD + swz(r, mcol >> 3)) = pack8(m);
                *reinterpret_cast<uint4 *>(bufD + swz(r, (mcol >> 3) + 1)) = pack8(m + 8);
                *reinterpret_cast<uint4 *>(bufE + swz(r, mcol >> 3)) = make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4 *>(bufE + swz(r, (mcol >> 3) + 1)) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        named_barrier(bar, kPrepThreads);
        // ---- N = D' E  (M = 64, N = 64, K = 64)
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id = idesc_bf16(64, 64, false, true);
            const uint32_t a = smem_u32(bufD), b = smem_u32(bufE);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_bf16(tmem, smem_desc(a + 32 * k, 16, 1024), smem_desc(b + 2048 * k, kTile, 1024),
                         id, k > 0);
            mma_commit(&sm.mma_bar);
        }
        if ((bad = unit_wait(&sm.mma_bar, mph, warp, bar, bad))) break;
        mph ^= 1;
        tc_fence_after();
        // N over E.  M = 64 layout: row 16 q + l in TMEM lane 32 q + l (l < 16);
        // the 16x256b shape hands every lane two rows' column pairs (the m8n8
        // fragment layout), which stmatrix writes.  Matrix m of an x4 group is
        // (row half m & 1, column group n + m / 2), its row k addressed by lane 8 m + k.
        const int fr = 16 * q4 + 8 * ((lane >> 3) & 1) + (lane & 7), fg = lane >> 4;
        {
            uint32_t y[32];
            tmem_ld16x256b_x8(tmem + lane_base, y);
            tmem_ld_wait();
#pragma unroll
            for (int n = 0; n < 8; n += 2)
                stmatrix_x4(bufE + swz(fr, n + fg),
                            pack_bf16(__uint_as_float(y[4 * n]), __uint_as_float(y[4 * n + 1])),
                            pack_bf16(__uint_as_float(y[4 * n + 2]), __uint_as_float(y[4 * n + 3])),
                            pack_bf16(__uint_as_float(y[4 * n + 4]), __uint_as_float(y[4 * n + 5])),
                            pack_bf16(__uint_as_float(y[4 * n + 6]), __uint_as_float(y[4 * n + 7])));
        }
        fence_proxy_async_smem();
        tc_fence_before();
        named_barrier(bar, kPrepThreads);
        // ---- Y = N D'  (M = 64, N = 64, K = 64)
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id = idesc_bf16(64, 64, false, true);
            const uint32_t a = smem_u32(bufE), b = smem_u32(bufD);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_bf16(tmem, smem_desc(a + 32 * k, 16, 1024), smem_desc(b + 2048 * k, kTile, 1024),
                         id, k > 0);
            mma_commit(&sm.mma_bar);
        }
        if ((bad = unit_wait(&sm.mma_bar, mph, warp, bar, bad))) break;
        mph ^= 1;
        tc_fence_after();
        // ---- T = D' - Y;  T diag(b) in place of D' (then copied to the
        // slot), T diag(b e^gamma) into ab; D' read with ldmatrix in the same
        // fragment layout as Y.
        {
            uint32_t y[32];
            tmem_ld16x256b_x8(tmem + lane_base, y);
            tmem_ld_wait();
            const int cp = 2 * (lane & 3);  // this lane's column pair within a group
#pragma unroll
            for (int n = 0; n < 8; n += 2) {
                uint32_t d[4], tb[4], tbg[4];
                ldmatrix_x4(bufD + swz(fr, n + fg), d[0], d[1], d[2], d[3]);
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int c = 8 * (n + (m >> 1)) + cp;
                    const float2 bb = *reinterpret_cast<const float2 *>(sm.beta + c);
                    const float2 bgv = *reinterpret_cast<const float2 *>(sm.bg + c);
                    const float2 dv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&d[m]));
                    const int yi = 4 * (n + (m >> 1)) + 2 * (m & 1);
                    const float t0 = dv.x - __uint_as_float(y[yi]), t1 = dv.y - __uint_as_float(y[yi + 1]);
                    tb[m] = pack_bf16(t0 * bb.x, t1 * bb.y);
                    tbg[m] = pack_bf16(t0 * bgv.x, t1 * bgv.y);
                }
                stmatrix_x4(bufD + swz(fr, n + fg), tb[0], tb[1], tb[2], tb[3]);
                stmatrix_x4(sm.ab + swz(fr, n + fg), tbg[0], tbg[1], tbg[2], tbg[3]);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        named_barrier(bar, kPrepThreads);
        // ---- W^T = K^T (T diag(b e^gamma))^T  (M = 128 dk, N = 64, K = 64 tokens)
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id = idesc_bf16(128, 64, true, false);
            const uint32_t a = smem_u32(sm.kq), b = smem_u32(sm.ab);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_bf16(tmem, smem_desc(a + 2048 * k, 2 * kTile, 1024),
                         smem_desc(b + 32 * k, 16, 1024), id, k > 0);
            mma_commit(&sm.mma_bar);
        }
        if (tid == kCopier) {
            bulk_store(slot + kSlotTB, bufD, kTile);
            bulk_commit_group();
        }
        if ((bad = unit_wait(&sm.mma_bar, mph, warp, bar, bad))) break;
        mph ^= 1;
        tc_fence_after();
        // W^T staged (16 KB) in K atom 0 + Q atom 0 (both dead), then copied.
        {
            uint8_t *const wt = sm.kq;
            const int wr = row;
            float y[32];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                tmem_ld32f(tmem + lane_base + 32 * hf, y);
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
                    *reinterpret_cast<uint4 *>(wt + swz(wr, 4 * hf + cc)) = pack8(y + 8 * cc);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        named_barrier(bar, kPrepThreads);
        if (tid == kCopier) {
            bulk_store(slot + kSlotWT, sm.kq, 2 * kTile);
            bulk_commit_group();
            // The recurrence may be waiting for this item: publish at once
            // (the copier waits for its copies here; the next item's tiles
            // are issued after it).
            if (flags) publish_item(flags + (size_t)ch * Hv + h, epoch);
        }
        if (!kLoop) break;
    }
    if (tid == kCopier) bulk_wait_group<0>();  // shared memory must outlive the copies
    if (bad && tid == 0) atomicCAS(err, (int)kErrNone, (int)kErrTimeout);  // (the first error stays)
    tc_fence_before();
    named_barrier(bar, kPrepThreads);
    if (warp == 0) tmem_dealloc(tmem, kPrepTmemCols);
    if (tid == 0) {  // (the memory may hold something else next)
        mbar_inval(&sm.tma_bar);
        mbar_inval(&sm.mma_bar);
    }
}

__global__ void __launch_bounds__(kPrepThreads, kPrepCtasPerSm)
gdn_prep_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const float *__restrict__ g, const float *__restrict__ beta,
                const int *__restrict__ chunk_off, const int4 *__restrict__ table,
                uint8_t *__restrict__ slots, float *__restrict__ gl, int *__restrict__ err, int N,
                int Hk, int Hv) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    PrepSmem &sm = *reinterpret_cast<PrepSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    // Launched as a programmatic dependent of the chunk table kernel: let the
    // recurrence kernel be scheduled once all of this grid is placed, then
    // wait for the table.
    griddep_launch_dependents();
    griddep_wait();
    if ((int)blockIdx.x >= chunk_off[N]) return;
    const int item = blockIdx.x * Hv + blockIdx.y;
    prep_unit<false>(sm, &tm_q, &tm_k, g, beta, chunk_off, table, slots, gl, err, N, Hk, Hv,
                     threadIdx.x, 1, 2, item, 1, item + 1, nullptr, 0u, true);
}

// ------------------------------------------------------------------ kernel 3
constexpr int kChainThreads = 448;  // 14 warps: 0 loads, 1 MMAs, 2-9 state, 10-13 output
constexpr int kStateThreads = 256;
constexpr int kOutThreads = 128;

struct alignas(1024) ChainStage {  // 1024-aligned: the tiles are 128-byte-swizzle atoms
    uint8_t k[2 * kTile];   // K [64 tokens][128 dk] as two 64-column atoms
    uint8_t q[2 * kTile];   // diag(e^gamma) Q, likewise
    uint8_t v[2 * kTile];   // V [64 tokens][128 dv]
    uint8_t wt[2 * kTile];  // W^T [128 dk][64 tokens], MN-major B image
    uint8_t tb[kTile];      // T diag(b)
    uint8_t p[kTile];       // P = M o Q K^T
    float egdec[2 * C];     // e^{gamma_t}, then e^{gamma_L - gamma_t}
};

// The snapshot stores stage 8 warps x 8 KB in the K, Q~, V, W^T tiles.
static_assert(offsetof(ChainStage, q) == 2 * kTile && offsetof(ChainStage, v) == 4 * kTile &&
                  offsetof(ChainStage, wt) == 6 * kTile && offsetof(ChainStage, tb) == 8 * kTile,
              "snapshot staging needs K, Q~, V, W^T contiguous");

struct ChainSmem {
    ChainStage st[2];
    uint8_t ostage[3][C * D * 2];  // output tiles [64 tokens][128 dv] bf16, for TMA stores
    uint64_t full[2];              // stage loaded (TMA transaction count)
    uint64_t empty[2];             // stage consumed (MMA commit + state threads)
    uint64_t s16_ready;            // state threads: -S0 (bf16) and pre-scaled S in TMEM
    uint64_t dt_ready;             // state threads: Delta^T copies in TMEM
    uint64_t o_free[2];            // output threads: output accumulator (by chunk parity) read
    uint64_t d_done;               // MMA: Delta^T complete
    uint64_t s_done;               // MMA: state update complete
    uint64_t o_done[2];            // MMA: output accumulator (by chunk parity) complete
    uint64_t fin;                  // MMA: everything issued has completed
    uint32_t tmem;
    int abort;
    int issued;
};

constexpr uint32_t kStageBytes = 10 * kTile + 512;  // K, Q~, V, W^T, T diag b, P, e^gamma/dec
constexpr int kPrefetch = 3;  // chunks pulled into L2 ahead of the two staged ones
// Below this the state's running scale factor is folded back into the
// stored state (keeps 1 / sigma far from fp32 overflow).
constexpr float kRenorm = 1.0e-12f;
// TMEM columns of the recurrence kernel.  D = U^T then Delta^T (fp32); O =
// S0 Q~^T + Delta^T P^T (fp32, two buffers by chunk parity, so that the
// output warps read one while the next chunk's output accumulates); NS = -S0
// as bf16 pairs (the A operand of two MMAs, two buffers); S = the fp32 state;
// DT and DTS = Delta^T and Delta^T diag(e^{gamma_L - gamma}) as bf16 pairs
// (A operands).  NS is double-buffered by chunk parity: chunk c's S0 Q~^T may
// be issued after its state update, i.e. after the state warps have written
// chunk c + 1's -S0.
constexpr uint32_t kColD = 0, kColO = 64, kColNS = 192, kColS = 320, kColDT = 448,
                   kColDTS = 480;

__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&x)[64]) {
    uint32_t r[32];
    tmem_ld32(taddr, r);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(r[i]);
    tmem_ld32(taddr + 32, r);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; ++i) x[32 + i] = __uint_as_float(r[i]);
}

// Stores 64 state values of one row: -x as 32 bf16 pairs into NS and
// scale * x as fp32 into S.
__device__ __forceinline__ void store_state(uint32_t t_ns, uint32_t t_s, const float (&x)[64],
                                            float scale) {
    uint32_t r[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = pack_bf16(-x[2 * i], -x[2 * i + 1]);
    tmem_st32(t_ns, r);
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(scale * x[i]);
    tmem_st32(t_s, r);
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(scale * x[32 + i]);
    tmem_st32(t_s + 32, r);
}

// A state warp's 32 rows x 64 columns of sigma S^ (the state after chunk c)
// into snapshot plane z of `map` ([planes, 128 dv, 128 dk] fp32).  Once o_done shows
// chunk c's MMAs complete, the stage's K, Q~, V and W^T tiles (64 KB, 8 KB a
// warp) are dead: the rows are staged there as two [32][32] fp32 boxes
// (128-byte swizzle: conflict-free) and stored by TMA, so the global writes
// bypass the load/store pipe that the chain's waits go through (row-per-
// thread stores would touch 32 lines per instruction).  S^ is read from TMEM
// again: it stays put until this warp's next dt_ready.  The stage goes back
// to the producer once the stores have read it.  Out of line
// and rarely taken, so the chain loop stays small in the instruction cache.
// False when a bounded wait ran out.
__device__ __noinline__ bool store_state_rows(ChainSmem &sm, const CUtensorMap *map, uint32_t t_s,
                                              float sigma, int c, int z) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (!warp_wait_lean(&sm.o_done[c & 1], (c >> 1) & 1, &sm.abort)) return false;
    uint8_t *stg = sm.st[c & 1].k + (warp - 2) * kTile;
#pragma unroll 1
    for (int b = 0; b < 2; ++b) {
        uint32_t r[32];
        tmem_ld32(t_s + 32 * b, r);
        tmem_ld_wait();
        uint8_t *box = stg + b * (kTile / 2);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            *reinterpret_cast<float4 *>(box + swz(lane, i)) = make_float4(
                sigma * __uint_as_float(r[4 * i]), sigma * __uint_as_float(r[4 * i + 1]),
                sigma * __uint_as_float(r[4 * i + 2]), sigma * __uint_as_float(r[4 * i + 3]));
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        const int x = 64 * ((warp - 2) >> 2), y = 32 * (warp & 3);
        tma_store_3d(map, x, y, z, stg);
        tma_store_3d(map, x + 32, y, z, stg + kTile / 2);
        bulk_commit_group();
        bulk_wait_group_read<0>();
    }
    __syncwarp();
    mbar_arrive(&sm.empty[c & 1]);
    return true;
}

// kSnaps: the instantiation that writes chunk-boundary snapshots (a separate
// instantiation keeps the snapshot code out of the plain kernel's hot loop).
// kLinear: the instantiation for the chunk-parallel scan that runs the
// recurrence's linear part alone: the initial state is the identity and U is
// zero, so the final state is the product of the chunks' transition matrices
// (the output it writes is not used).  kNoOut: only the final state is
// wanted (the scan's group passes): no output MMAs, output warps or Q~/P loads.
// The recurrence for (sequence, value head) number `bid` of the sorted order.
// Warps: 0 loads, 1 MMAs, kS0..kS0+7 state, kS0+8..kS0+11 output, any other
// idle.  kFused: inside the persistent kernel that also runs prep (below):
// the loads of chunk c wait for its ready flag, and the chunk decay comes
// from the stage instead of the workspace.
// kMulti (fused kernel only): the CTA runs value head h = bid over every
// sequence in turn, as one stream of chunks 0 .. chunk_off[N] - 1 (the
// recurrence restarts from each sequence's initial state at its first chunk
// and stores its final state after its last).  Otherwise: one (sequence,
// value head) recurrence, order[bid / Hv] and bid % Hv.
template <bool kSnaps, bool kLinear, bool kNoOut, int kS0, bool kFused, bool kMulti = false>
__device__ __forceinline__ void chain_role(
    ChainSmem &sm, int bid, const CUtensorMap *tm_k, const CUtensorMap *tm_v,
    const CUtensorMap *tm_o, const CUtensorMap *tm_s, const int *__restrict__ chunk_off,
    const int *__restrict__ order, const int4 *__restrict__ table,
    const uint8_t *__restrict__ slots, const float *__restrict__ gl,
    const float *__restrict__ h0, __nv_bfloat16 *__restrict__ out, float *__restrict__ hT,
    float *__restrict__ snaps, int snap_stride, const int *__restrict__ snap_off,
    int *__restrict__ err, int N, int Hk, int Hv, const unsigned *__restrict__ flags,
    int c_flagged = 0) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    static_assert(!kMulti || (kFused && !kSnaps && !kLinear && !kNoOut), "kMulti: fused only");
    griddep_wait();  // a programmatic dependent of prep: wait for its slots
    const int n = kMulti ? 0 : order[bid / Hv], h = kMulti ? bid : bid % Hv;
    const int hk = h / (Hv / Hk);
    const int c_begin = kMulti ? 0 : chunk_off[n];
    const int nc = kMulti ? chunk_off[N] : chunk_off[n + 1] - c_begin;
    const size_t state_off = ((size_t)n * Hv + h) * D * D;  // (kMulti: per sequence)
    const int n_thr = kFused ? (int)blockDim.x : kChainThreads;
    // kMulti: final state = initial state for every empty sequence of head h
    // (one warp per sequence).
    auto copy_empty_states = [&]() {
        if (!hT || (chunk_off[N] == 0 && *err != kErrNone)) return;
        for (int m = warp; m < N; m += n_thr / 32) {
            if (chunk_off[m + 1] != chunk_off[m]) continue;
            const size_t off = ((size_t)m * Hv + h) * D * D;
            for (int i = lane; i < D * D / 4; i += 32) {
                const float4 x = h0 ? reinterpret_cast<const float4 *>(h0 + off)[i]
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
                reinterpret_cast<float4 *>(hT + off)[i] = x;
            }
        }
    };
    // Epilogue warps: TMEM quadrant q, state or output row j.
    const int q = warp & 3;
    const int j = 32 * q + lane;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;

    if (kMulti && nc == 0) {
        copy_empty_states();
        return;
    }
    if (nc == 0) {
        // Empty sequence (or a rejected chunk table): final state = initial state.
        if (hT && !(chunk_off[N] == 0 && *err != kErrNone)) {
            for (int i = tid; i < D * D / 4; i += kFused ? (int)blockDim.x : kChainThreads) {
                const float4 x = h0 ? reinterpret_cast<const float4 *>(h0 + state_off)[i]
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
                reinterpret_cast<float4 *>(hT + state_off)[i] = x;
            }
        }
        return;
    }

    if (tid == 0) {
        prefetch_tensormap(tm_k);
        prefetch_tensormap(tm_v);
        prefetch_tensormap(tm_o);
        if (kSnaps) prefetch_tensormap(tm_s);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1 + kStateThreads);
        }
        mbar_init(&sm.s16_ready, kStateThreads);
        mbar_init(&sm.dt_ready, kStateThreads);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.o_free[b], kOutThreads);
            mbar_init(&sm.o_done[b], 1);
        }
        mbar_init(&sm.d_done, 1);
        mbar_init(&sm.s_done, 1);
        mbar_init(&sm.fin, 1);
        sm.abort = 0;
        sm.issued = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&sm.tmem, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem;

    if (warp < 2) {
    if (warp == 0) {
        // ---------------- producer: TMA tiles and the prep kernel's slot;
        // chunks kPrefetch ahead are pulled into L2 so that a stage's loads
        // hit L2 when the stage frees up.  The whole warp runs the loop and one
        // elected lane issues each copy.
        {
            // A sequence's chunks are consecutive 64-token windows.
            const int seq_tok0 = table[c_begin].y;
            auto prefetch = [&](int c) {
                if (lane != 0) return;
                const int ch = c_begin + c;
                const int tok0 = kMulti ? table[ch].y : seq_tok0 + C * c;
                tma_prefetch_3d(tm_k, 0, hk, tok0);
                tma_prefetch_3d(tm_k, 64, hk, tok0);
                tma_prefetch_3d(tm_v, 0, h, tok0);
                tma_prefetch_3d(tm_v, 64, h, tok0);
                bulk_prefetch_l2(slots + ((size_t)ch * Hv + h) * kSlotBytes, kSlotBytes);
            };
            #pragma unroll 1
            for (int c = 2; c < min(nc, 2 + kPrefetch); ++c) prefetch(c);
            __syncwarp();
            #pragma unroll 1
            for (int c = 0; c < nc; ++c) {
                const int s = c & 1;
                // (in the fused kernel the chunk's ready flag first: its
                // acquire overlaps the wait for the stage)
                if (kFused && c >= c_flagged &&
                    !wait_ready(flags + (size_t)(c_begin + c) * Hv + h, &sm.abort))
                    break;
                if (c >= 2 && !warp_wait_lean(&sm.empty[s], ((c >> 1) + 1) & 1, &sm.abort)) break;
                const int ch = c_begin + c;
                const int tok0 = kMulti ? table[ch].y : seq_tok0 + C * c;
                if (kDebug) {
                    // The chunk's table entry agrees with the sequence's.
                    const int4 te = table[ch];
                    if (!(ch < chunk_off[N] && te.y == tok0 && te.z >= 1 && te.z <= C &&
                          te.x >= 0 && te.x < N && (kMulti || te.x == n))) {
                        if (lane == 0) {
                            debug_fail(err, kErrIndex);
                            sm.abort = 1;
                        }
                        break;
                    }
                }
                ChainStage &st = sm.st[s];
                uint64_t *bar = &sm.full[s];
                const uint8_t *slot = slots + ((size_t)ch * Hv + h) * kSlotBytes;
                // One elected lane issues the stage's copies (per-copy
                // elections cost code the instruction cache has to hold).
                if (elect_one_sync()) {
                    mbar_arrive_expect_tx(bar, kStageBytes - (kNoOut ? 3 * kTile : 0) -
                                                   (kLinear ? 3 * kTile : 0));
                    tma_load_3d(st.k, tm_k, 0, hk, tok0, bar);
                    tma_load_3d(st.k + kTile, tm_k, 64, hk, tok0, bar);
                    if (!kLinear) {
                        tma_load_3d(st.v, tm_v, 0, h, tok0, bar);
                        tma_load_3d(st.v + kTile, tm_v, 64, h, tok0, bar);
                        bulk_load(st.tb, slot + kSlotTB, kTile, bar);
                    }
                    bulk_load(st.wt, slot + kSlotWT, 2 * kTile, bar);
                    if (!kNoOut) {
                        bulk_load(st.p, slot + kSlotP, kTile, bar);
                        bulk_load(st.q, slot + kSlotQ, 2 * kTile, bar);
                    }
                    bulk_load(st.egdec, slot + kSlotEG, 512, bar);
                }
                if (lane == 0) sm.issued = c + 1;
                if (c + 2 + kPrefetch - 1 < nc && c >= 1) prefetch(c + 2 + kPrefetch - 1);
                __syncwarp();
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer: the whole warp runs this loop with
        // identical values (descriptors stay warp-uniform) and one lane,
        // elected once per group, issues the group's tcgen05 instructions.
        // U^T for chunk c + 1 is issued right after chunk c's last MMAs, so it
        // runs while the state warps prepare chunk c + 1's S0.
        {
            constexpr uint32_t id_u = idesc_bf16(128, 64, true, false);
            constexpr uint32_t id_w = idesc_bf16(128, 64, false, true);
            constexpr uint32_t id_q = idesc_bf16(128, 64, false, false);
            constexpr uint32_t id_qn = idesc_bf16(128, 64, false, false, true);  // A negated
            constexpr uint32_t id_s = idesc_bf16(128, 64, false, true);
            // D = U^T = V^T (T diag b)^T             [M=128 dv, N=64, K=64 tokens]
            auto issue_u = [&](int c) -> bool {
                const int s = c & 1;
                if (!warp_wait_lean(&sm.full[s], (c >> 1) & 1, &sm.abort)) return false;
                tc_fence_after();
                ChainStage &st = sm.st[s];
                const uint64_t d_v = smem_desc(smem_u32(st.v), kTile, 1024);
                const uint64_t d_tb = smem_desc(smem_u32(st.tb), 16, 1024);
if (!kLinear && elect_one_sync()) {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_bf16(tmem + kColD, d_v + 128 * k, d_tb + 2 * k, id_u, k > 0);
                }
                __syncwarp();
                return true;
            };
            bool ok = issue_u(0);
            #pragma unroll 1
            for (int c = 0; ok && c < nc; ++c) {
                const int s = c & 1;
                ChainStage &st = sm.st[s];
                // Base descriptors; a k-step moves the start address only
                // (the 14-bit address field cannot carry: smem < 256 KB).
                const uint64_t d_wt = smem_desc(smem_u32(st.wt), kTile, 1024);
                const uint64_t d_q = smem_desc(smem_u32(st.q), 16, 1024);
                const uint64_t d_k = smem_desc(smem_u32(st.k), kTile, 1024);
                const uint64_t d_p = smem_desc(smem_u32(st.p), 16, 1024);
                const uint32_t ns = kColNS + 64 * (c & 1);
                const uint32_t ob = kColO + 64 * (c & 1);
                if (!warp_wait_lean(&sm.s16_ready, c & 1, &sm.abort)) break;
                tc_fence_after();
                // D += (-S0) W^T  ->  Delta^T            [M=128 dv, N=64, K=128 dk]
if (elect_one_sync()) {
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        mma_bf16_ta(tmem + kColD, tmem + ns + 8 * k, d_wt + 128 * k, id_w,
                                    !kLinear || k > 0);
                    mma_commit(&sm.d_done);
                }
                __syncwarp();
                // O = S0 Q~^T (A = -S0, negated)         [M=128 dv, N=64, K=128 dk]
                // into this chunk's output buffer, free once the output warps
                // have read chunk c - 2's (they have two chunk steps for it, so
                // the wait normally returns at once).  Each MMA group has one
                // copy of its code: the issuing warp's loop has to stay small
                // enough for the instruction cache, or its MMAs issue at
                // instruction-fetch speed.
                if (!kNoOut && c >= 2 &&
                    !warp_wait_lean(&sm.o_free[c & 1], ((c >> 1) - 1) & 1, &sm.abort))
                    break;
                tc_fence_after();
if (!kNoOut && elect_one_sync()) {
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        mma_bf16_ta(tmem + ob, tmem + ns + 8 * k,
                                    d_q + (k / 4) * (kTile / 16) + 2 * (k % 4), id_qn, k > 0);
                }
                __syncwarp();
                if (!warp_wait_lean(&sm.dt_ready, c & 1, &sm.abort)) break;
                tc_fence_after();
                // S^ += (Delta^T diag(e^{gamma_L - gamma}) / sigma) K   [M=128, N=128, K=64]
                // as two N = 64 halves (an N = 128 MMA with A in TMEM runs
                // several times slower than two N = 64 ones).
if (elect_one_sync()) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        mma_bf16_ta(tmem + kColS, tmem + kColDTS + 8 * k, d_k + 128 * k, id_s, 1);
                        mma_bf16_ta(tmem + kColS + 64, tmem + kColDTS + 8 * k,
                                    d_k + (kTile >> 4) + 128 * k, id_s, 1);
                    }
                    mma_commit(&sm.s_done);
                }
                __syncwarp();
                // O += Delta^T P^T                       [M=128 dv, N=64, K=64 tokens]
if (elect_one_sync()) {
#pragma unroll
                    for (int k = 0; k < (kNoOut ? 0 : 4); ++k)
                        mma_bf16_ta(tmem + ob, tmem + kColDT + 8 * k, d_p + 2 * k, id_q, 1);
                    mma_commit(&sm.o_done[c & 1]);
                    mma_commit(&sm.empty[s]);
                }
                __syncwarp();
                if (c + 1 < nc) ok = issue_u(c + 1);
            }
            mma_commit_w(&sm.fin);
        }
    }
    } else if (warp < kS0 + 8) {  // (warps below kS0 took the branch above)
        // ---------------- state warps 2-9: row j, half h2 of the state's
        // columns (and of Delta's 64 tokens).  The state is kept in TMEM as
        // S^ with S = sigma S^: the chunk decay e^{gamma_L} folds into sigma,
        // and 1 / sigma into the Delta operand of the update, so the fp32
        // state is only rewritten when sigma gets small (renormalisation).
        // E3: Delta^T -> bf16 A operands; E6: S -> -S0 (bf16).
        const int h2 = (warp - kS0) >> 2;
        const uint32_t t_ns = tmem + lane_base + kColNS + 32 * h2;  // + 64 * (chunk & 1)
        const uint32_t t_s = tmem + lane_base + kColS + 64 * h2;
        float sigma = 1.f;
        bool ok = true;
        // Snapshot countdown and plane (no division in the loop).
        int snap_left = snap_stride, snap_z = kSnaps ? snap_off[n] * Hv + h : 0;
        // (kMulti) the state's sequence: its initial and final state plane
        size_t st_off = kMulti ? ((size_t)table[c_begin].x * Hv + h) * D * D : state_off;
        {
            float x[64];
#pragma unroll
            for (int c = 0; c < 64; c += 4) {
                float4 v4 = h0 ? *reinterpret_cast<const float4 *>(
                                     h0 + st_off + (size_t)j * D + 64 * h2 + c)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
                if (kLinear) {
                    const int k0 = 64 * h2 + c;
                    v4 = make_float4(j == k0, j == k0 + 1, j == k0 + 2, j == k0 + 3);
                }
                x[c] = v4.x; x[c + 1] = v4.y; x[c + 2] = v4.z; x[c + 3] = v4.w;
            }
            store_state(t_ns, t_s, x, 1.f);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&sm.s16_ready);
        }
        #pragma unroll 1
        for (int c = 0; ok && c < nc; ++c) {
            // (kMulti) the next chunk's entry: a sequence starts there when it
            // is that sequence's chunk 0 (read now, used after two waits)
            const int4 te_next = (kMulti && c + 1 < nc) ? table[c_begin + c + 1]
                                                         : make_int4(0, 0, 0, 1);
            const float *dec = sm.st[c & 1].egdec + C;
            // e^{gamma_L} of chunk c (in the fused kernel from the stage, which
            // holds e^{gamma_t} with gamma constant past the chunk's end)
            const float decay_g = kFused ? 1.f : gl[(size_t)(c_begin + c) * Hv + h];
            bool snap_here = false;
            if (kSnaps) {
                snap_here = --snap_left == 0 || c == nc - 1;
                if (snap_left == 0) snap_left = snap_stride;
            }
            if (!(ok = warp_wait_lean(&sm.d_done, c & 1, &sm.abort))) break;
            tc_fence_after();
            const float decay = kFused ? sm.st[c & 1].egdec[C - 1] : decay_g;
            float sigma_next = sigma * decay;
            if (!(sigma_next >= kRenorm)) {
                // Fold sigma_next into S^ (sigma becomes 1).  G6 of the previous
                // chunk has completed (its s_done was observed) and this
                // chunk's G6 waits for dt_ready, so S^ is ours to rewrite.
                float x[64];
                tmem_ld64(t_s, x);
                uint32_t r[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(sigma_next * x[i]);
                tmem_st32(t_s, r);
#pragma unroll
                for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(sigma_next * x[32 + i]);
                tmem_st32(t_s + 32, r);
                sigma_next = 1.f;
            }
            const float inv = 1.f / sigma_next;
            {
                uint32_t r[32];
                tmem_ld32(tmem + lane_base + kColD + 32 * h2, r);
                tmem_ld_wait();
                uint32_t pd[16], ps[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float d0 = __uint_as_float(r[2 * i]), d1 = __uint_as_float(r[2 * i + 1]);
                    const float2 dv = *reinterpret_cast<const float2 *>(dec + 32 * h2 + 2 * i);
                    pd[i] = pack_bf16(d0, d1);
                    const float2 pr = mul2(mul2(make_float2(d0, d1), dv), make_float2(inv, inv));
                    ps[i] = pack_bf16(pr.x, pr.y);
                }
                tmem_st16(tmem + lane_base + kColDT + 16 * h2, pd);
                tmem_st16(tmem + lane_base + kColDTS + 16 * h2, ps);
                tmem_st_wait();
            }
            sigma = sigma_next;
            tc_fence_before();
            mbar_arrive(&sm.dt_ready);
            if (!snap_here) mbar_arrive(&sm.empty[c & 1]);  // else after the snapshot
            if (!(ok = warp_wait_lean(&sm.s_done, c & 1, &sm.abort))) break;
            tc_fence_after();
            {
                float x[64];
                tmem_ld64(t_s, x);
                if (c == nc - 1 || te_next.w == 0) {
                    if (hT) {
                        float *dst = hT + st_off + (size_t)j * D + 64 * h2;
#pragma unroll
                        for (int i = 0; i < 64; i += 4)
                            *reinterpret_cast<float4 *>(dst + i) =
                                make_float4(sigma * x[i], sigma * x[i + 1], sigma * x[i + 2],
                                            sigma * x[i + 3]);
                    }
                    if (kMulti && c + 1 < nc) {
                        // The next sequence starts from its own initial state
                        // (in place of the hand-off; S^ and this parity's -S0
                        // are free as they are for the hand-off).
                        st_off = ((size_t)te_next.x * Hv + h) * D * D;
#pragma unroll
                        for (int i = 0; i < 64; i += 4) {
                            const float4 v4 = h0 ? *reinterpret_cast<const float4 *>(
                                                       h0 + st_off + (size_t)j * D + 64 * h2 + i)
                                                 : make_float4(0.f, 0.f, 0.f, 0.f);
                            x[i] = v4.x; x[i + 1] = v4.y; x[i + 2] = v4.z; x[i + 3] = v4.w;
                        }
                        store_state(t_ns + 64 * ((c + 1) & 1), t_s, x, 1.f);
                        tmem_st_wait();
                        sigma = 1.f;
                        tc_fence_before();
                        mbar_arrive(&sm.s16_ready);
                    }
                } else {
                    // -S0 of chunk c + 1 for the MMAs (the hand-off).
                    uint32_t r[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float2 pr = mul2(make_float2(x[2 * i], x[2 * i + 1]),
                                               make_float2(-sigma, -sigma));
                        r[i] = pack_bf16(pr.x, pr.y);
                    }
                    tmem_st32(t_ns + 64 * ((c + 1) & 1), r);
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(&sm.s16_ready);
                }
            }
            if (snap_here) {
                if (!(ok = store_state_rows(sm, tm_s, t_s, sigma, c, snap_z))) break;
                snap_z += Hv;
            }
        }
        if (kSnaps && lane == 0) bulk_wait_group<0>();
    } else if (warp < kS0 + 12) {
        // ---------------- output warps: o_t = S0 (e^{gamma_t} q_t) +
        // (Delta^T P^T)_t for this warp's 32 value dims, read from this
        // chunk's output accumulator with the 16x256b TMEM shape (the m8n8
        // fragment layout) and written transposed with stmatrix into a
        // [64 tokens][128 dv] tile held as two 128-byte-swizzled halves, then
        // stored by TMA (a short last chunk, whose tile would reach into the
        // next sequence, is copied out row by row instead).
        const bool leader = (warp == kS0 + 8 && lane == 0);
        const int hh = q >> 1;                  // dv half of this warp's rows
        const int k8 = lane & 7, d8 = lane >> 3; // stmatrix row and matrix of this lane
#pragma unroll 1
        for (int c = 0; c < (kNoOut ? 0 : nc); ++c) {
            const int4 e = table[c_begin + c];
            const int tok0 = e.y, L = e.z;
            if (!warp_wait_lean(&sm.o_done[c & 1], (c >> 1) & 1, &sm.abort)) break;
            tc_fence_after();
            uint32_t r[2][32];
            tmem_ld16x256b_x8(tmem + lane_base + kColO + 64 * (c & 1), r[0]);
            tmem_ld16x256b_x8(tmem + lane_base + (16u << 16) + kColO + 64 * (c & 1), r[1]);
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(&sm.o_free[c & 1]);
            uint8_t *stg = sm.ostage[c % 3];
            if (leader) bulk_wait_group_read<2>();  // the stores from chunk c - 3 have read it
            named_barrier(1, kOutThreads);
            // Matrix d8 of a group: value dims 32 (q & 1) + 8 d8 .. + 7 of half
            // hh (16-byte chunk 4 (q & 1) + d8 of a 128-byte row); row k8 is
            // token 8 g + k8.
            uint8_t *tile = stg + hh * kTile;
            const uint32_t chunk = 4 * (q & 1) + d8;
#pragma unroll
            for (int g = 0; g < C / 8; ++g)
                stmatrix_x4_trans(tile + swz(8 * g + k8, chunk),
                                  pack_bf16(__uint_as_float(r[0][4 * g]), __uint_as_float(r[0][4 * g + 1])),
                                  pack_bf16(__uint_as_float(r[0][4 * g + 2]), __uint_as_float(r[0][4 * g + 3])),
                                  pack_bf16(__uint_as_float(r[1][4 * g]), __uint_as_float(r[1][4 * g + 1])),
                                  pack_bf16(__uint_as_float(r[1][4 * g + 2]), __uint_as_float(r[1][4 * g + 3])));
            if (L == C) {
                fence_proxy_async_smem();
                named_barrier(1, kOutThreads);
                if (leader) {
                    tma_store_3d(tm_o, 0, h, tok0, stg);
                    tma_store_3d(tm_o, 64, h, tok0, stg + kTile);
                    bulk_commit_group();
                }
            } else {
                named_barrier(1, kOutThreads);
                // Rows t < L: 16 chunks of 16 bytes each, un-swizzled.
                const int tid_o = tid - (kS0 + 8) * 32;
                for (int idx = tid_o; idx < L * 16; idx += kOutThreads) {
                    const int t = idx >> 4, cc = idx & 15;
                    const uint4 v = *reinterpret_cast<const uint4 *>(stg + (cc >> 3) * kTile +
                                                                     swz(t, cc & 7));
                    *reinterpret_cast<uint4 *>(out + ((size_t)(tok0 + t) * Hv + h) * D + 8 * cc) = v;
                }
            }
        }
        if (leader) bulk_wait_group<0>();
    }
    __syncthreads();
    if (kMulti && !sm.abort) copy_empty_states();
    if (sm.abort) {
        if (tid == 0) {
            atomicCAS(err, (int)kErrNone, (int)kErrTimeout);  // (the first error stays)
            // Let loads still in flight land before the CTA leaves.
            for (int c = max(0, sm.issued - 2); c < sm.issued; ++c)
                mbar_wait(&sm.full[c & 1], (c >> 1) & 1, 200000000ll);
        }
    }
    if (tid == 32) mbar_wait(&sm.fin, 0, 200000000ll);  // MMA warp's final commit
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

template <bool kSnaps, bool kLinear = false, bool kNoOut = false>
__global__ void __launch_bounds__(kChainThreads, 1)
gdn_chain_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                 const __grid_constant__ CUtensorMap tm_o, const __grid_constant__ CUtensorMap tm_s,
                 const int *__restrict__ chunk_off, const int *__restrict__ order,
                 const int4 *__restrict__ table, const uint8_t *__restrict__ slots,
                 const float *__restrict__ gl, const float *__restrict__ h0,
                 __nv_bfloat16 *__restrict__ out,
                 float *__restrict__ hT, float *__restrict__ snaps, int snap_stride,
                 const int *__restrict__ snap_off, int *__restrict__ err, int N, int Hk, int Hv) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    ChainSmem &sm = *reinterpret_cast<ChainSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    chain_role<kSnaps, kLinear, kNoOut, 2, false>(sm, blockIdx.x, &tm_k, &tm_v, &tm_o, &tm_s,
                                                  chunk_off, order, table, slots, gl, h0, out, hT,
                                                  snaps, snap_stride, snap_off, err, N, Hk, Hv,
                                                  nullptr);
}

// ------------------------------------------------------------------ fused prep + recurrence
// One persistent cooperative launch, one CTA of 512 threads per SM (up to 128
// registers a thread: the recurrence's warps compile as in the separate
// kernel).  CTAs below n_chain run a recurrence each (warps 0-13, 14-15
// idle): of one (sequence, value head), or (kMulti) of one value head over
// every sequence in turn.  The others run four prep units each over the
// (chunk, value head) items in the prep order, each unit publishing an item's
// ready flag as soon as its slot is written, and the recurrence waits for the
// flag of each chunk before loading it.  Prep never waits for the recurrence
// and all CTAs are resident (cooperative launch), so every wait ends.  Prep
// runs on the SMs the recurrence leaves idle, during the recurrence instead
// of before it.
constexpr int kFusedThreads = kPrepUnits * kPrepThreads;
constexpr int kLocalChunks = kPrepUnits;  // chunks each recurrence preps itself (one round)
static_assert(kFusedThreads >= kChainThreads, "the recurrence's warps fit the fused CTA");
constexpr size_t kPrepUnitBytes = sizeof(PrepSmem);  // a multiple of 1024 (alignas)
constexpr size_t kPrepCtaBytes = kPrepUnits * kPrepUnitBytes;  // a prep CTA's units
constexpr size_t kFusedSmemBytes =
    (sizeof(ChainSmem) > kPrepCtaBytes ? sizeof(ChainSmem) : kPrepCtaBytes) + 1024;
static_assert(kFusedSmemBytes <= 232448, "fused kernel shared memory");
static_assert(kPrepUnits * kPrepTmemCols <= 512, "prep units' TMEM");
static_assert(1 + 2 * kPrepUnits <= 16, "prep units' named barriers");

// kMulti: n_chain = Hv recurrences, each over all sequences in turn (value
// head h = blockIdx.x), and prep in the chunks' own order, which is then the
// order the recurrences take them in.  For batches whose N x Hv recurrences
// would not leave SMs for prep.
template <bool kMulti>
__global__ void __launch_bounds__(kFusedThreads, 1)
gdn_fused_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                 const float *__restrict__ g, const float *__restrict__ beta,
                 const int *__restrict__ chunk_off, const int *__restrict__ order,
                 const int4 *__restrict__ table, uint8_t *__restrict__ slots,
                 float *__restrict__ gl, const float *__restrict__ h0,
                 __nv_bfloat16 *__restrict__ out, float *__restrict__ hT, int *__restrict__ err,
                 unsigned *__restrict__ flags, const int *__restrict__ porder, int N, int Hk,
                 int Hv, int n_chain, int n_items) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    griddep_wait();  // (a programmatic dependent of the chunk table kernel)
    const int u = threadIdx.x / kPrepThreads;
    if ((int)blockIdx.x < n_chain) {
        // The recurrence's first kLocalChunks chunks are prepped here, one
        // per unit, before it starts (the prep CTAs begin with the chunks
        // after them): the recurrence then waits for its own first chunks
        // only, not for the first round of every prep unit of the grid.  (Two
        // rounds here avoid the wait for that round, whose items run twice as
        // long as later ones, but start the recurrence later and slow its
        // steps while more prep runs beside them: slower at 4000 tokens.)
        const int n = kMulti ? 0 : order[blockIdx.x / Hv];
        const int h = kMulti ? (int)blockIdx.x : (int)blockIdx.x % Hv;
        const int c_begin = kMulti ? 0 : chunk_off[n];
        const int n_local = min((kMulti ? chunk_off[N] : chunk_off[n + 1]) - c_begin, kLocalChunks);
#pragma unroll 1
        for (int c = u; c < n_local; c += kPrepUnits) {
            const int item = (c_begin + c) * Hv + h;
            prep_unit<false>(*reinterpret_cast<PrepSmem *>(base + u * kPrepUnitBytes), &tm_q,
                             &tm_k, g, beta, chunk_off, table, slots, gl, err, N, Hk, Hv,
                             threadIdx.x - u * kPrepThreads, 1 + u, 1 + kPrepUnits + u, item, 1,
                             item + 1, nullptr, 0u, false);
        }
        fence_proxy_async_global();  // (this thread's slot writes, before the loads of them)
        __syncthreads();
        chain_role<false, false, false, 2, true, kMulti>(
            *reinterpret_cast<ChainSmem *>(base), blockIdx.x, &tm_k, &tm_v, &tm_o, &tm_o,
            chunk_off, order, table, slots, gl, h0, out, hT, nullptr, 1, nullptr, err, N, Hk, Hv,
            flags, n_local);
    } else {
        // Skip what the recurrences prep themselves: in the prep order (by
        // position in the sequence) the first sum_n min(chunks_n, kLocalChunks)
        // chunks; (kMulti) the first kLocalChunks chunks.
        __shared__ int s_first;
        if (threadIdx.x == 0) {
            int s = 0;
            if (kMulti) {
                s = min(chunk_off[N], kLocalChunks);
            } else {
                for (int m = 0; m < N; ++m) s += min(chunk_off[m + 1] - chunk_off[m], kLocalChunks);
            }
            s_first = s;
        }
        __syncthreads();
        // The units' first two rounds in order, then items drawn from the
        // ticket after the flags, in the prep order.
        const int pcta = blockIdx.x - n_chain, n_units = kPrepUnits * (gridDim.x - n_chain);
        prep_unit<true>(*reinterpret_cast<PrepSmem *>(base + u * kPrepUnitBytes), &tm_q, &tm_k, g,
                        beta, chunk_off, table, slots, gl, err, N, Hk, Hv,
                        threadIdx.x - u * kPrepThreads, 1 + u, 1 + kPrepUnits + u,
                        s_first * Hv + kPrepUnits * pcta + u, n_units, n_items, flags, 1u, false,
                        kMulti ? nullptr : porder, flags + n_items, s_first * Hv + 2 * n_units);
    }
}

// ------------------------------------------------------------------ chunk-parallel scan
// The chunk step is affine in the state, S_{c+1} = S_c M_c + B_c (with
// M_c = e^{gamma_L} I - W^T diag(e^{gamma_L - gamma}) K and
// B_c = U^T diag(e^{gamma_L - gamma}) K), and composes by
// (M, B) then (M', B') = (M M', B M' + B').  A sequence is cut into groups
// of L chunks (pseudo-sequences that the prep and recurrence kernels treat
// like sequences): the recurrence from a zero state gives each group's B,
// the kLinear recurrence (identity state, U = 0) its M, the combine kernel
// below carries the state across groups, and a last recurrence pass from
// each group's initial state writes the outputs.

// One CTA of 1024 threads.  Checks cu_seqlens like the chunk table kernel,
// then goff[n] = groups before sequence n (G_n = ceil(chunks_n / L), 0 for an
// empty sequence) and cu2 = the pseudo-sequences' token offsets, padded with
// T up to n2 + 1 entries.  A malformed cu_seqlens gives cu2[0] = 1, which the
// chunk table kernel rejects (the whole call is then a no-op).
__global__ void __launch_bounds__(1024)
gdn_scan_split_kernel(const int32_t *__restrict__ cu, int N, int64_t T, int L, int n2,
                      int32_t *__restrict__ cu2, int *__restrict__ goff) {
    __shared__ int s_scan[1024];
    __shared__ int s_carry, s_bad;
    const int tid = threadIdx.x;
    if (tid == 0) {
        s_carry = 0;
        s_bad = (cu[0] != 0 || (int64_t)cu[N] != T) ? 1 : 0;
    }
    __syncthreads();
    for (int base = 0; base < N; base += 1024) {
        const int n = base + tid;
        int gn = 0;
        if (n < N) {
            const int len = cu[n + 1] - cu[n];
            if (len < 0) s_bad = 1;
            const int nch = len > 0 ? (len + C - 1) / C : 0;
            gn = (nch + L - 1) / L;
        }
        s_scan[tid] = gn;
        __syncthreads();
        for (int off = 1; off < 1024; off <<= 1) {
            const int x = tid >= off ? s_scan[tid - off] : 0;
            __syncthreads();
            s_scan[tid] += x;
            __syncthreads();
        }
        if (n < N) {
            const int first = s_carry + s_scan[tid] - gn;
            goff[n] = first;
            for (int gi = 0; gi < gn && first + gi < n2; ++gi)
                cu2[first + gi] = cu[n] + C * L * gi;
        }
        __syncthreads();
        if (tid == 1023) s_carry += s_scan[1023];
        __syncthreads();
    }
    const int total = s_carry;
    if (tid == 0) goff[N] = total;
    for (int i = total + tid; i <= n2; i += 1024) cu2[i] = (int32_t)T;
    __syncthreads();
    if (tid == 0 && (s_bad || total > n2)) cu2[0] = 1;
}

// Carries the state across the groups of each (sequence, value head):
// Hbuf[group] = the state entering the group, S <- S M_g + B_g, and the
// final state into hT.  Rows are independent, so CTA y owns rows
// 16y..16y+15 (grid N Hv x 8, 128 threads).  Warp w computes columns
// 32w..32w+31; lane l a 4 x 4 tile (rows 4 (l / 8).., columns 32w + 4 (l % 8)..),
// reading S transposed and M from shared memory (two 16-byte loads per 16
// FMAs).  The next group's M is fetched with cp.async into the other buffer
// while this one is used.  fp32 throughout.  Does nothing when the chunk
// table kernel rejected cu_seqlens.
constexpr int kCombineRows = 16;
constexpr int kCombineThreads = 128;

__device__ __forceinline__ void combine_fetch_m(float *dst, const float *src, int tid) {
    const uint32_t d = smem_u32(dst);
#pragma unroll 4
    for (int i = tid; i < D * D / 4; i += kCombineThreads)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d + 16 * i),
                     "l"(src + 4 * i)
                     : "memory");
    asm volatile("cp.async.commit_group;" ::: "memory");
}

__global__ void __launch_bounds__(kCombineThreads)
gdn_scan_combine_kernel(const int *__restrict__ goff, const float *__restrict__ h0,
                        const float *__restrict__ mbuf, const float *__restrict__ bbuf,
                        float *__restrict__ hbuf, float *__restrict__ hT,
                        const int *__restrict__ err, int Hv) {
    extern __shared__ __align__(16) float cm_smem[];
    float *ms = cm_smem;                   // M of two groups [2][128][128]
    float *st = cm_smem + 2 * D * D;       // S transposed [128 k][16 rows]
    if (*err != kErrNone) return;
    const int n = blockIdx.x / Hv, h = blockIdx.x % Hv;
    const int tid = threadIdx.x, w = tid >> 5, l = tid & 31;
    const int r0 = 4 * (l >> 3), c0 = 32 * w + 4 * (l & 7);
    const int row0 = kCombineRows * blockIdx.y + r0;
    float s[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 x = h0 ? *reinterpret_cast<const float4 *>(
                                  h0 + ((size_t)(n * Hv + h) * D + row0 + i) * D + c0)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
        s[i][0] = x.x; s[i][1] = x.y; s[i][2] = x.z; s[i][3] = x.w;
    }
    const int g_begin = goff[n], g_end = goff[n + 1];
    if (g_begin < g_end) combine_fetch_m(ms, mbuf + (size_t)(g_begin * Hv + h) * D * D, tid);
#pragma unroll 1
    for (int gi = g_begin; gi < g_end; ++gi) {
        const size_t plane = (size_t)gi * Hv + h;
        const float *mcur = ms + ((gi - g_begin) & 1) * D * D;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            *reinterpret_cast<float4 *>(hbuf + (plane * D + row0 + i) * D + c0) =
                make_float4(s[i][0], s[i][1], s[i][2], s[i][3]);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) st[(c0 + jj) * kCombineRows + r0 + i] = s[i][jj];
        }
        if (gi + 1 < g_end) {
            combine_fetch_m(ms + ((gi + 1 - g_begin) & 1) * D * D, mbuf + (plane + Hv) * D * D,
                            tid);
            asm volatile("cp.async.wait_group 1;" ::: "memory");
        } else {
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 b = *reinterpret_cast<const float4 *>(
                bbuf + (plane * D + row0 + i) * D + c0);
            s[i][0] = b.x; s[i][1] = b.y; s[i][2] = b.z; s[i][3] = b.w;
        }
#pragma unroll 4
        for (int k = 0; k < D; ++k) {
            const float4 a = *reinterpret_cast<const float4 *>(st + k * kCombineRows + r0);
            const float4 m = *reinterpret_cast<const float4 *>(mcur + k * D + c0);
            const float av[4] = {a.x, a.y, a.z, a.w}, mv[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) s[i][jj] = fmaf(av[i], mv[jj], s[i][jj]);
        }
        __syncthreads();
    }
    if (hT) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            *reinterpret_cast<float4 *>(hT + ((size_t)(n * Hv + h) * D + row0 + i) * D + c0) =
                make_float4(s[i][0], s[i][1], s[i][2], s[i][3]);
    }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// [T, H, 128] bf16 tensor, boxes of 64 features x 1 head x 64 tokens, 128-byte swizzle.
bool encode_thd(CUtensorMap *map, const void *base, int64_t T, int H) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)(T > 0 ? T : 1)};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
    // 64-feature boxes, 128-byte swizzle: the MMA operand layout for loads,
    // and the bank-conflict-free staging layout of the output stores.
    const cuuint32_t box[3] = {64u, 1, (cuuint32_t)C};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Snapshots as a [slots Hv, 128 dv, 128 dk] fp32 tensor; boxes of 32 dk x
// 32 dv rows, 128-byte swizzle (the staging layout of the stores).
bool encode_states(CUtensorMap *map, float *base, int64_t planes) {
    auto enc = tensor_map_encoder();
    if (!enc || planes < 1 || planes > (int64_t)UINT32_MAX) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)D, (cuuint64_t)planes};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)D * D * 4};
    const cuuint32_t box[3] = {32u, 32u, 1u};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launch configuration with programmatic stream serialization (the kernel may
// be scheduled before the previous one in the stream completes; it calls
// griddep_wait before touching that kernel's output); `attr` must outlive
// the launch call.
cudaLaunchConfig_t pdl_config(dim3 grid, unsigned threads, size_t smem, cudaStream_t stream,
                              bool pdl, cudaLaunchAttribute *attr) {
    attr->id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr->val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = pdl ? attr : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cfg;
}

// Per-call timing (gdn_chunk_prefill_timed): caller-created events recorded
// on the launching stream before the chunk table, after it, after prep and
// after the recurrence (or the fused kernel); null when the call is not
// timed.  Nothing about it outlives the call.
struct Timing {
    cudaEvent_t ev[4];
    int *fused;  // set to 1 when prep and the recurrence ran as one launch
};

void time_mark(const Timing *tm, int i, cudaStream_t s) {
    if (tm) cudaEventRecord(tm->ev[i], s);
}

// (0 separate kernels, 1 fused, 2 fused with one recurrence per value head)
void time_fused(const Timing *tm, int fused) {
    if (tm && tm->fused) *tm->fused = fused;
}

// Fused path mode (gdn_prefill_fused_mode): 0 off, 1 whenever it can run,
// 2 when the cost model below expects it to be faster, 3 the variant with one
// recurrence per value head whenever it can run.
std::atomic<int> g_fused_mode{2};

constexpr int kMaxDevices = 64;

}  // namespace

int prefill_fused_mode(int mode) {
    if (mode >= 0 && mode <= 3) return g_fused_mode.exchange(mode);
    return g_fused_mode.load();
}

size_t prefill_tc_workspace_size(const gdn_problem &p) { return ws_layout(p).total; }

int64_t prefill_tc_snapshot_slots(const gdn_problem &p, int snap_stride) {
    return (ws_layout(p).max_chunks + snap_stride - 1) / snap_stride + p.num_seqs;
}

bool prefill_tc_supported(const gdn_problem &p) {
    return p.qkv_dtype == GDN_BF16 && p.head_dim_k == D && p.head_dim_v == D;
}

namespace {

struct TcMaps {
    CUtensorMap tq, tk, tv, to;
};

struct TcPtrs {
    int *err, *chunk_off, *snap_off, *order;
    int4 *table;
    float *gl;
    uint8_t *slots;
    unsigned *flags;
    int *porder;
};

TcPtrs tc_ptrs(const WsLayout &w, void *workspace) {
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    return {reinterpret_cast<int *>(ws + w.hdr), reinterpret_cast<int *>(ws + w.chunk_off),
            reinterpret_cast<int *>(ws + w.snap_off), reinterpret_cast<int *>(ws + w.order),
            reinterpret_cast<int4 *>(ws + w.table), reinterpret_cast<float *>(ws + w.gl),
            ws + w.tiles, reinterpret_cast<unsigned *>(ws + w.flags),
            reinterpret_cast<int *>(ws + w.porder)};
}

bool encode_maps(const gdn_problem &p, const void *q, const void *k, const void *v, void *out,
                 TcMaps &m) {
    if (p.total_tokens == 0) {
        memset(&m, 0, sizeof(m));
        return true;
    }
    return encode_thd(&m.tq, q, p.total_tokens, p.num_k_heads) &&
           encode_thd(&m.tk, k, p.total_tokens, p.num_k_heads) &&
           encode_thd(&m.tv, v, p.total_tokens, p.num_v_heads) &&
           encode_thd(&m.to, out, p.total_tokens, p.num_v_heads);
}

// The chunk table kernel (with `zero_flags`, it also clears the ready flags and
// the prep ticket of the fused kernel).
// zero_flags: also clear the fused kernel's flags and ticket and write its
// prep order; orders: the recurrences' sequence order and that prep order
// (the fused kernel with one recurrence per value head reads neither).
gdn_status launch_table(const gdn_problem &p, const WsLayout &w, const TcPtrs &t,
                        const int32_t *cu, int snap_stride, bool zero_flags, cudaStream_t stream,
                        const Timing *tm, bool orders = true) {
    time_mark(tm, 0, stream);
    gdn_chunk_table_kernel<<<1, 1024, 0, stream>>>(
        cu, p.num_seqs, p.total_tokens, w.max_chunks, snap_stride, t.err, t.chunk_off, t.snap_off,
        orders ? t.order : nullptr, t.table, t.flags,
        zero_flags ? (int)(w.max_chunks * p.num_v_heads) + 1 : 0,
        zero_flags && orders ? t.porder : nullptr);
    if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
    time_mark(tm, 1, stream);
    return GDN_OK;
}

// Prep (a programmatic dependent of the chunk table kernel).
gdn_status launch_prep(const gdn_problem &p, const WsLayout &w, const TcPtrs &t, const TcMaps &m,
                       const float *g, const float *beta, cudaStream_t stream, bool pdl,
                       const Timing *tm) {
    if (p.total_tokens > 0) {
        const size_t smem = sizeof(PrepSmem) + 1024;
        if (cudaFuncSetAttribute(gdn_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess)
            return GDN_ERR_CUDA;
        cudaLaunchAttribute attr;
        const cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)w.max_chunks, p.num_v_heads),
                                                  kPrepThreads, smem, stream, pdl, &attr);
        if (cudaLaunchKernelEx(&cfg, gdn_prep_kernel, m.tq, m.tk, g, beta,
                               (const int *)t.chunk_off, (const int4 *)t.table, t.slots, t.gl,
                               t.err, p.num_seqs, p.num_k_heads, p.num_v_heads) != cudaSuccess)
            return GDN_ERR_CUDA;
    }
    time_mark(tm, 2, stream);
    return GDN_OK;
}

gdn_status launch_table_prep(const gdn_problem &p, const WsLayout &w, const TcPtrs &t,
                             const TcMaps &m, const float *g, const float *beta,
                             const int32_t *cu, int snap_stride, cudaStream_t stream, bool pdl,
                             const Timing *tm = nullptr) {
    const gdn_status st = launch_table(p, w, t, cu, snap_stride, false, stream, tm);
    return st != GDN_OK ? st : launch_prep(p, w, t, m, g, beta, stream, pdl, tm);
}

// The recurrence kernel over the chunk table of `p` (a programmatic
// dependent of the kernel before it when `pdl`).
template <bool kSnaps, bool kLinear, bool kNoOut = false>
gdn_status launch_chain(const gdn_problem &p, const TcPtrs &t, const TcMaps &m,
                        const CUtensorMap &ts, const float *h0, void *out, float *hT,
                        float *snaps, int snap_stride, cudaStream_t stream, bool pdl) {
    const size_t smem = sizeof(ChainSmem) + 1024;
    auto chain = gdn_chain_kernel<kSnaps, kLinear, kNoOut>;
    if (cudaFuncSetAttribute(chain, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return GDN_ERR_CUDA;
    cudaLaunchAttribute attr;
    const cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)p.num_seqs * p.num_v_heads),
                                              kChainThreads, smem, stream, pdl, &attr);
    if (cudaLaunchKernelEx(&cfg, chain, m.tk, m.tv, m.to, ts, (const int *)t.chunk_off,
                           (const int *)t.order, (const int4 *)t.table, (const uint8_t *)t.slots,
                           (const float *)t.gl, h0, static_cast<__nv_bfloat16 *>(out), hT, snaps,
                           snap_stride, (const int *)t.snap_off, t.err, p.num_seqs,
                           p.num_k_heads, p.num_v_heads) != cudaSuccess)
        return GDN_ERR_CUDA;
    return GDN_OK;
}

// SMs the fused kernel can run on (one CTA each) on the current device, or 0
// when it cannot be used there: no cooperative launch, or less than one CTA
// per SM.  Looked up once per device and variant (the kernel's shared-memory
// attribute is set with that device current), under a lock.
template <bool kMulti>
int fused_grid() {
    static std::mutex mu;
    static int grid_of[kMaxDevices];
    static bool known[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return 0;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (known[dev]) return grid_of[dev];
    int sms = 0, coop = 0, blocks = 0, grid = 0;
    cudaFuncAttributes fa;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess ||
        cudaFuncSetAttribute(gdn_fused_kernel<kMulti>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kFusedSmemBytes) != cudaSuccess ||
        cudaFuncGetAttributes(&fa, gdn_fused_kernel<kMulti>) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, gdn_fused_kernel<kMulti>,
                                                      kFusedThreads, kFusedSmemBytes) !=
            cudaSuccess) {
        cudaGetLastError();
    } else if (coop && blocks >= 1) {
        grid = sms;
    }
    grid_of[dev] = grid;
    known[dev] = true;
    return grid;
}

// Whether the fused kernel should beat the separate ones, from measured rates
// on this GPU: a prep item (chunk, value head) takes kPrepItemUs on one of the
// kPrepUnits units of a CTA in either kernel, a recurrence chunk step
// kChainStepUs.  Fused: prep on the SMs the recurrences leave, the
// recurrence following (it cannot finish before its last chunk is prepped),
// after kFusedStartUs: each recurrence's own first round of prep and the
// prep units' first round, whose code runs cold on every SM.  Separate: prep
// on every SM, then the recurrence.  The longest sequence is estimated as
// T / N tokens (as long as T for one sequence).  (At 16/48 heads this puts
// the crossover between 1472 and 2000 tokens of one sequence; measured it
// lies between 1000 and 1408: separate against fused 50.8 / 51.9 µs at 1000
// tokens, 61.1 / 60.1 at 1408, 81.6 / 71.3 at 2000, 30.3 / 38.5 at 352.)
constexpr double kPrepItemUs = 8.0, kChainStepUs = 1.3, kFusedStartUs = 21.0;
bool fused_pays(const gdn_problem &p, int grid) {
    const int64_t n_chain = (int64_t)p.num_seqs * p.num_v_heads;
    if (n_chain + 16 > grid) return false;
    const int64_t chunks = (p.total_tokens + C - 1) / C + p.num_seqs - 1;
    const int64_t items = chunks * p.num_v_heads;
    const double chain = kChainStepUs * (double)((p.total_tokens / p.num_seqs + C - 1) / C);
    const int64_t units_f = kPrepUnits * (grid - n_chain), units_s = kPrepCtasPerSm * (int64_t)grid;
    const double prep_f = kPrepItemUs * (double)((items + units_f - 1) / units_f);
    const double prep_s = kPrepItemUs * (double)((items + units_s - 1) / units_s);
    return std::max(prep_f, chain) + kFusedStartUs < prep_s + chain + 5.0;
}

// Whether the kMulti fused kernel should beat the separate kernels, from
// rates measured on GB300 (16/48 heads, d = 128, L2 flushed; each fits the
// measured times of 2-2000 sequences within about 10 %), in µs:
//   separate: prep 5 + 12.5 per wave of 5 x SMs items; then the (sequence,
//     value head) recurrences, ceil(N Hv / SMs) waves of the mean sequence's
//     chunks, each chunk max(1.25, 0.019 x the recurrences running at once
//     - 0.3) (HBM-bound when many run), plus 2 per wave and 5;
//   kMulti: 20 + per chunk of the batch max(1.25, the prep time of its Hv
//     items on the 4 (SMs - Hv) units at 12.5 each).
// The host does not know the lengths (cu_seqlens is on the device): the
// chunk count is taken as ceil(T / 64) + (N - 1) / 4, and the longest
// sequence as the mean one, which understates the separate recurrence of a
// batch of unequal lengths.  kMulti needs an estimate 5 % below the other.
bool multi_pays(const gdn_problem &p, int grid) {
    const int64_t N = p.num_seqs, Hv = p.num_v_heads;
    if (Hv + 16 > grid || N < 2) return false;
    const double chunks = (double)((p.total_tokens + C - 1) / C) + (double)(N - 1) / 4.0;
    const double items = chunks * (double)Hv;
    const double prep_s = 5.0 + 12.5 * items / (double)(kPrepCtasPerSm * grid);
    const int64_t pairs = N * Hv;
    const double waves = (double)((pairs + grid - 1) / grid);
    const double conc = (double)std::min<int64_t>(pairs, grid);
    const double mean_chunks = (double)((p.total_tokens / N + C - 1) / C);
    const double step_s = std::max(1.25, 0.019 * conc - 0.3);
    const double chain_s = 5.0 + waves * (mean_chunks * step_s + 2.0);
    const double step_m =
        std::max(1.25, 12.5 * (double)Hv / (double)(kPrepUnits * (grid - Hv)));
    const double multi = 20.0 + chunks * step_m;
    return multi < 0.95 * (prep_s + chain_s);
}

}  // namespace

// The kernels a prefill of `p` runs: 0 the separate prep and recurrence
// kernels, 1 the fused kernel with one recurrence per (sequence, value head),
// 2 the fused kernel with one recurrence per value head over all sequences;
// `grid` and `grid_m` are the SMs the two fused variants can use (0: they
// cannot run).  Fused with one recurrence per (sequence, value head) when
// they leave 16 SMs for prep (mode 2: and its cost model prefers it), else
// the per-head variant (mode 1: when the first does not fit, mode 2: when its
// cost model prefers it, mode 3: whenever it fits).
int prefill_path(const gdn_problem &p, int grid, int grid_m, int mode) {
    if (p.total_tokens == 0 || mode == 0 || p.num_seqs <= 0) return 0;
    const bool fits = (int64_t)p.num_seqs * p.num_v_heads + 16 <= grid;
    if (mode != 3 && grid > 0 && (mode == 1 ? fits : fused_pays(p, grid))) return 1;
    if (fits && mode == 1) return 0;
    if (grid_m > 0 && (mode == 2 ? multi_pays(p, grid_m) : p.num_v_heads + 16 <= grid_m))
        return 2;
    return 0;
}

namespace {

// Chunk table, then the fused kernel: prep and the recurrence in one launch.
// False when the launch was refused (the caller then runs the separate
// kernels; the chunk table is already in place).
bool launch_fused(const gdn_problem &p, const WsLayout &w, const TcPtrs &t, const TcMaps &m,
                  const float *g, const float *beta, const float *h0, void *out, float *hT,
                  int grid, bool multi, cudaStream_t stream, bool pdl) {
    // Cooperative (every CTA resident, so the waits on ready flags end) and,
    // unless the call is timed, a programmatic dependent of the chunk table
    // kernel (its CTAs are placed and set up while the table is written; they
    // wait for it before reading it).  Without the second attribute if the
    // driver refuses the pair.
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kFusedThreads);
    cfg.dynamicSmemBytes = kFusedSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    const int n_chain = multi ? p.num_v_heads : p.num_seqs * p.num_v_heads;
    const int n_items = (int)(w.max_chunks * p.num_v_heads);
    auto kernel = multi ? gdn_fused_kernel<true> : gdn_fused_kernel<false>;
    for (int na = pdl ? 2 : 1; na >= 1; --na) {
        cfg.numAttrs = na;
        if (cudaLaunchKernelEx(&cfg, kernel, m.tq, m.tk, m.tv, m.to, g, beta,
                               (const int *)t.chunk_off, (const int *)t.order,
                               (const int4 *)t.table, t.slots, t.gl, h0,
                               static_cast<__nv_bfloat16 *>(out), hT, t.err, t.flags,
                               (const int *)t.porder, p.num_seqs, p.num_k_heads, p.num_v_heads,
                               n_chain, n_items) == cudaSuccess)
            return true;
        cudaGetLastError();
    }
    return false;
}

}  // namespace

gdn_status launch_prefill_tc(const gdn_problem &p, const void *q, const void *k, const void *v,
                             const float *g, const float *beta, const int32_t *cu,
                             const float *h0, void *out, float *hT, float *snaps,
                             int snap_stride, cudaStream_t stream, void *const *events,
                             int *fused) {
    Timing timing;
    const Timing *tm = nullptr;
    if (events) {
        for (int i = 0; i < 4; ++i) timing.ev[i] = static_cast<cudaEvent_t>(events[i]);
        timing.fused = fused;
        tm = &timing;
    }
    time_fused(tm, 0);
    if (p.num_seqs == 0) return GDN_OK;
    const WsLayout w = ws_layout(p);
    const TcPtrs t = tc_ptrs(w, p.workspace);
    TcMaps m;
    if (!encode_maps(p, q, k, v, out, m)) return GDN_ERR_CUDA;
    // The prep and recurrence launches overlap their predecessor's tail
    // (programmatic dependent launch), except in a timed call, whose events
    // sit between them.
    const bool pdl = tm == nullptr;
    // (sequence x value head) recurrences that leave SMs for prep: the fused
    // kernel.
    const int mode = prefill_fused_mode(-1);
    const bool plain = snaps || p.total_tokens == 0 || mode == 0;
    const int grid = plain ? 0 : fused_grid<false>();
    const int grid_m = plain ? 0 : fused_grid<true>();
    const int path = plain ? 0 : prefill_path(p, grid, grid_m, mode);
    const bool multi = path == 2;
    if (path != 0) {
        gdn_status st = launch_table(p, w, t, cu, 0, true, stream, tm, !multi);
        if (st != GDN_OK) return st;
        time_mark(tm, 2, stream);  // (no separate prep launch)
        if (launch_fused(p, w, t, m, g, beta, h0, out, hT, multi ? grid_m : grid, multi, stream,
                         pdl)) {
            time_mark(tm, 3, stream);
            time_fused(tm, multi ? 2 : 1);
            return GDN_OK;
        }
        // (the launch was refused: the separate kernels, with the sequence
        // order the chunk table left out for the per-head variant)
        if (multi && (st = launch_table(p, w, t, cu, 0, false, stream, tm)) != GDN_OK) return st;
        st = launch_prep(p, w, t, m, g, beta, stream, false, tm);
        if (st != GDN_OK) return st;
        st = launch_chain<false, false>(p, t, m, m.to, h0, out, hT, nullptr, 1, stream, false);
        if (st != GDN_OK) return st;
        time_mark(tm, 3, stream);
        return GDN_OK;
    }
    gdn_status st =
        launch_table_prep(p, w, t, m, g, beta, cu, snaps ? snap_stride : 0, stream, pdl, tm);
    if (st != GDN_OK) return st;
    CUtensorMap ts = m.to;
    if (snaps && !encode_states(&ts, snaps,
                                prefill_tc_snapshot_slots(p, snap_stride) * p.num_v_heads))
        return GDN_ERR_CUDA;
    st = snaps ? launch_chain<true, false>(p, t, m, ts, h0, out, hT, snaps, snap_stride, stream, pdl)
               : launch_chain<false, false>(p, t, m, ts, h0, out, hT, nullptr, 1, stream, pdl);
    if (st != GDN_OK) return st;
    time_mark(tm, 3, stream);
    return GDN_OK;
}

gdn_status launch_prefill_tc_prep_only(const gdn_problem &p, const void *q, const void *k,
                                      const float *g, const float *beta, const int32_t *cu,
                                      cudaStream_t stream) {
    if (p.num_seqs == 0) return GDN_OK;
    const WsLayout w = ws_layout(p);
    const TcPtrs t = tc_ptrs(w, p.workspace);
    TcMaps m;
    // (v and out are not touched by the table and prep kernels: their maps
    // are built over q)
    if (!encode_maps(p, q, k, q, const_cast<void *>(q), m)) return GDN_ERR_CUDA;
    return launch_table_prep(p, w, t, m, g, beta, cu, 0, stream, false);
}

void prefill_tc_slot_layout(const gdn_problem &p, int64_t *layout) {
    const WsLayout w = ws_layout(p);
    layout[0] = (int64_t)w.tiles;
    layout[1] = kSlotBytes;
    layout[2] = kSlotWT;
    layout[3] = kSlotTB;
    layout[4] = kSlotP;
    layout[5] = kSlotQ;
    layout[6] = kSlotEG;
    layout[7] = kSlotDEC;
}

namespace {

// Workspace of the chunk-parallel scan: the prefill workspace of the problem
// whose sequences are the groups (n2 of them at most), then the groups'
// token offsets, the group offsets of each sequence, and the groups' M, B and
// initial states ([n2 Hv, 128, 128] fp32 each).
struct ScanLayout {
    gdn_problem p2;
    WsLayout w2;
    size_t cu2, goff, mbuf, bbuf, hbuf, total;
    int n2;
};

ScanLayout scan_layout(const gdn_problem &p, int L) {
    ScanLayout sl;
    const int64_t chunks = (p.total_tokens + C - 1) / C + p.num_seqs;
    sl.n2 = (int)std::min<int64_t>(p.num_seqs + (chunks + L - 1) / L, INT32_MAX / 2);
    sl.p2 = p;
    sl.p2.num_seqs = sl.n2;
    sl.w2 = ws_layout(sl.p2);
    const size_t plane = (size_t)sl.n2 * p.num_v_heads * D * D * 4;
    sl.cu2 = align_up(sl.w2.total, 256);
    sl.goff = align_up(sl.cu2 + 4 * ((size_t)sl.n2 + 1), 256);
    sl.mbuf = align_up(sl.goff + 4 * ((size_t)p.num_seqs + 1), 1024);
    sl.bbuf = sl.mbuf + plane;
    sl.hbuf = sl.bbuf + plane;
    sl.total = sl.hbuf + plane;
    return sl;
}

}  // namespace

size_t prefill_scan_workspace_size(const gdn_problem &p, int chunks_per_group) {
    return scan_layout(p, chunks_per_group).total;
}

int prefill_scan_auto_group(const gdn_problem &p) {
    // SM count of the current device, looked up once per device.
    static std::atomic<int> sms_of[kMaxDevices];
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevices) {
        sms = sms_of[dev].load();
        if (sms == 0) {
            if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
                sms = 148;
            sms_of[dev].store(sms);
        }
    } else {
        cudaGetLastError();
    }
    // Enough groups that groups x value heads about fills the SMs once.
    const int64_t chunks = (p.total_tokens + C - 1) / C + p.num_seqs;
    const int64_t groups = std::max<int64_t>(1, sms / std::max(1, p.num_v_heads));
    return (int)std::max<int64_t>(4, (chunks + groups - 1) / groups);
}

gdn_status launch_prefill_scan(const gdn_problem &p, int L, const void *q, const void *k,
                               const void *v, const float *g, const float *beta,
                               const int32_t *cu, const float *h0, void *out, float *hT,
                               cudaStream_t stream) {
    if (p.num_seqs == 0) return GDN_OK;
    const ScanLayout sl = scan_layout(p, L);
    uint8_t *ws = static_cast<uint8_t *>(p.workspace);
    int32_t *cu2 = reinterpret_cast<int32_t *>(ws + sl.cu2);
    int *goff = reinterpret_cast<int *>(ws + sl.goff);
    float *mb = reinterpret_cast<float *>(ws + sl.mbuf);
    float *bb = reinterpret_cast<float *>(ws + sl.bbuf);
    float *hb = reinterpret_cast<float *>(ws + sl.hbuf);
    const TcPtrs t = tc_ptrs(sl.w2, p.workspace);
    TcMaps m;
    if (!encode_maps(p, q, k, v, out, m)) return GDN_ERR_CUDA;

    gdn_scan_split_kernel<<<1, 1024, 0, stream>>>(cu, p.num_seqs, p.total_tokens, L, sl.n2, cu2,
                                                   goff);
    if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
    gdn_status st = launch_table_prep(sl.p2, sl.w2, t, m, g, beta, cu2, 0, stream, false);
    if (st != GDN_OK) return st;
    // B of every group (the state from zero), then M (identity state, U = 0);
    // these passes write no output.
    st = launch_chain<false, false, true>(sl.p2, t, m, m.to, nullptr, out, bb, nullptr, 1, stream,
                                          true);
    if (st != GDN_OK) return st;
    st = launch_chain<false, true, true>(sl.p2, t, m, m.to, nullptr, out, mb, nullptr, 1, stream,
                                         true);
    if (st != GDN_OK) return st;
    const size_t smem = (size_t)(2 * D * D + kCombineRows * D) * 4;
    if (cudaFuncSetAttribute(gdn_scan_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return GDN_ERR_CUDA;
    gdn_scan_combine_kernel<<<dim3((unsigned)p.num_seqs * p.num_v_heads, D / kCombineRows),
                              kCombineThreads, smem, stream>>>(goff, h0, mb, bb, hb, hT, t.err, p.num_v_heads);
    if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
    // Outputs: every group from the state entering it.
    return launch_chain<false, false>(sl.p2, t, m, m.to, hb, out, nullptr, nullptr, 1, stream,
                                      false);
}

}  // namespace gdn
