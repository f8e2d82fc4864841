// prefill_tc.cu -- chunked prefill on the tcgen05 tensor cores (bf16 q/k/v,
// d_k = d_v = 128), as three launches on one stream:
//
//   1. gdn_chunk_table_kernel  one CTA: chunk offsets of every sequence, a
//      (sequence, first token, length) table of all chunks and the order in
//      which the recurrence CTAs take sequences (longest first).
//   2. gdn_prep_kernel         one CTA per (chunk, key head), all chunks at
//      once: the intra-chunk prep.  [K; Q] K^T on the tensor cores (one
//      M = 128 MMA gives K K^T and Q K^T), then for each value head of the
//      key head: gamma = cumsum(g), A_ti = b_t e^{gamma_t - gamma_i} (k_t . k_i)
//      for i < t, T = (I + A)^-1 by fp32 forward substitution, and the two
//      64 x 64 bf16 tiles the recurrence needs, T diag(b) and
//      P = M o Q K^T (M_ri = e^{gamma_r - gamma_i}, i <= r), written to the
//      workspace in the swizzled image of a shared-memory tile.
//   3. gdn_chain_kernel        one CTA per (sequence, value head): the
//      inter-chunk recurrence and the output.  The fp32 state S (dv x dk)
//      stays in tensor memory for the whole sequence; per chunk, with a bf16
//      copy of S0 in shared memory as the MMA operand:
//         U^T   = V^T (T diag b)^T                 (TMEM, fp32)
//         W^T   = K^T (T diag(b e^gamma))^T        (TMEM -> bf16 smem)
//         Delta^T = U^T - S0 W^T                   (accumulated onto U^T)
//         O1^T  = S0 Q^T,  O2^T = Delta^T P^T,  o_t = e^{gamma_t} O1 + O2
//         S     = e^{gamma_L} S0 + (diag(e^{gamma_L - gamma}) Delta)^T K
//      The next chunk's tiles arrive by TMA while the current one is used.
//
// The algorithm is the chunked (WY/UT) form of the Gated DeltaNet recurrence
// with chunk length 64, split into intra-chunk prep, inter-chunk state
// recurrence and output, as the page "cf-1.com" (section "三个优化", item 2
// "GDN prefill") describes its three kernels; that page keeps the state in
// mma accumulator registers on Turing, here it lives in Blackwell tensor
// memory.  Every MMA has M = 128 (the value or key dimension, or 64 keys
// plus 64 queries), so no tensor-core issue slot is half empty.
//
// Tokens past the end of a sequence inside its last chunk get b = 0 and
// g = 0, which zeroes their rows of W, U and Delta and keeps gamma_L at the
// last real token.
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "common.cuh"
#include "sm103.cuh"

namespace gdn {
namespace {

using namespace ptx;

constexpr int C = 64;           // chunk length
constexpr int D = 128;          // head dim (dk = dv)
constexpr int kTile = 8192;     // bytes of one 64 x 64 bf16 swizzled tile
constexpr int kPrepThreads = 192;
constexpr int kChainThreads = 128;
constexpr int kMaxSortSeqs = 4096;

enum DeviceError : int { kErrNone = 0, kErrCuSeqlens = 1, kErrTimeout = 2 };

// ------------------------------------------------------------------ workspace
struct WsLayout {
    size_t hdr, chunk_off, order, table, tiles, total;
    int64_t max_chunks;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

WsLayout ws_layout(const gdn_problem &p) {
    WsLayout w;
    w.max_chunks = (p.total_tokens + C - 1) / C + p.num_seqs;
    w.hdr = 0;
    w.chunk_off = 256;
    w.order = align_up(w.chunk_off + 4 * (size_t)(p.num_seqs + 1), 256);
    w.table = align_up(w.order + 4 * (size_t)p.num_seqs, 256);
    w.tiles = align_up(w.table + 16 * (size_t)w.max_chunks, 1024);
    w.total = w.tiles + (size_t)w.max_chunks * p.num_v_heads * 2 * kTile;
    return w;
}

// ------------------------------------------------------------------ kernel 1
// One CTA of 1024 threads.  chunk_off[n] = number of chunks before sequence n
// (chunk_off[N] = total), table[chunk] = {n, first token, length, index in
// sequence}, order = sequences by decreasing chunk count (stable), identity
// when N is large.  Malformed cu_seqlens (not starting at 0, decreasing, not
// ending at T, or more chunks than the workspace holds) record an error and
// make the whole call a no-op.
__global__ void __launch_bounds__(1024)
gdn_chunk_table_kernel(const int32_t *__restrict__ cu, int N, int64_t T, int64_t max_chunks,
                       int *__restrict__ err, int *__restrict__ chunk_off,
                       int *__restrict__ order, int4 *__restrict__ table) {
    __shared__ int s_scan[1024];
    __shared__ int s_carry;
    __shared__ int s_bad;
    const int tid = threadIdx.x;
    if (tid == 0) {
        s_carry = 0;
        s_bad = (cu[0] != 0 || (int64_t)cu[N] != T) ? 1 : 0;
        *err = kErrNone;
    }
    __syncthreads();
    for (int base = 0; base < N; base += 1024) {
        const int n = base + tid;
        int nch = 0;
        if (n < N) {
            const int len = cu[n + 1] - cu[n];
            if (len < 0) s_bad = 1;
            nch = len > 0 ? (len + C - 1) / C : 0;
        }
        s_scan[tid] = nch;
        __syncthreads();
        for (int off = 1; off < 1024; off <<= 1) {
            const int x = tid >= off ? s_scan[tid - off] : 0;
            __syncthreads();
            s_scan[tid] += x;
            __syncthreads();
        }
        if (n < N) chunk_off[n] = s_carry + s_scan[tid] - nch;
        __syncthreads();
        if (tid == 1023) s_carry += s_scan[1023];
        __syncthreads();
    }
    if (tid == 0) {
        if ((int64_t)s_carry > max_chunks) s_bad = 1;
        if (s_bad) *err = kErrCuSeqlens;
        chunk_off[N] = s_bad ? 0 : s_carry;
    }
    __syncthreads();
    if (s_bad) {
        for (int n = tid; n < N; n += 1024) chunk_off[n] = 0;
        for (int n = tid; n < N; n += 1024) order[n] = n;
        return;
    }
    const int total = s_carry;
    for (int ch = tid; ch < total; ch += 1024) {
        int lo = 0, hi = N - 1;  // last n with chunk_off[n] <= ch
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (chunk_off[mid] <= ch) lo = mid; else hi = mid - 1;
        }
        const int c = ch - chunk_off[lo];
        const int tok0 = cu[lo] + c * C;
        table[ch] = make_int4(lo, tok0, min(C, cu[lo + 1] - tok0), c);
    }
    for (int n = tid; n < N; n += 1024) {
        if (N > kMaxSortSeqs) {
            order[n] = n;
            continue;
        }
        const int mine = chunk_off[n + 1] - chunk_off[n];
        int rank = 0;
        for (int m = 0; m < N; ++m) {
            const int other = chunk_off[m + 1] - chunk_off[m];
            rank += (other > mine) || (other == mine && m < n);
        }
        order[rank] = n;
    }
}

// ------------------------------------------------------------------ kernel 2
struct PrepSmem {
    uint8_t kq[4 * kTile];            // atom 0: K rows 0-63, Q rows 64-127; atom 1 likewise
    float A[3][C][C + 4];             // A, then T, per value head of the round
    float gam[3][C];
    float beta[3][C];
    uint64_t tma_bar;
    uint64_t mma_bar;
    uint32_t tmem;
};

// Inclusive prefix sum of g over one chunk (lane holds tokens 2l, 2l+1),
// with g = 0 past the end of the sequence.  Optionally also b (0 past the
// end), e^{gamma_t} and e^{gamma_L - gamma_t}.  Called by one full warp.
__device__ __forceinline__ void chunk_gamma(const float *__restrict__ g, int tok0, int L, int Hv,
                                            int h, float *gam, float *beta_out,
                                            const float *__restrict__ beta, float *eg = nullptr,
                                            float *dec = nullptr) {
    const int lane = threadIdx.x & 31;
    const int t0 = 2 * lane, t1 = 2 * lane + 1;
    const float g0 = t0 < L ? g[(size_t)(tok0 + t0) * Hv + h] : 0.f;
    const float g1 = t1 < L ? g[(size_t)(tok0 + t1) * Hv + h] : 0.f;
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
}

__global__ void __launch_bounds__(kPrepThreads, 2)
gdn_prep_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const float *__restrict__ g, const float *__restrict__ beta,
                const int *__restrict__ chunk_off, const int4 *__restrict__ table,
                uint8_t *__restrict__ tiles, int *__restrict__ err, int N, int Hk, int Hv) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    PrepSmem &sm = *reinterpret_cast<PrepSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ch = blockIdx.x, hk = blockIdx.y;
    if (ch >= chunk_off[N]) return;
    const int4 e = table[ch];
    const int tok0 = e.y, L = e.z;
    const int G = Hv / Hk;

    if (tid == 0) {
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        mbar_init(&sm.tma_bar, 1);
        mbar_init(&sm.mma_bar, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&sm.tmem, 64);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem;
    if (tid == 0) {
        mbar_arrive_expect_tx(&sm.tma_bar, 4 * kTile);
        tma_load_3d(sm.kq + 0 * kTile, &tm_k, 0, hk, tok0, &sm.tma_bar);
        tma_load_3d(sm.kq + 1 * kTile, &tm_q, 0, hk, tok0, &sm.tma_bar);
        tma_load_3d(sm.kq + 2 * kTile, &tm_k, 64, hk, tok0, &sm.tma_bar);
        tma_load_3d(sm.kq + 3 * kTile, &tm_q, 64, hk, tok0, &sm.tma_bar);
    }
    bool bad = !mbar_wait(&sm.tma_bar, 0);
    if (tid == 0 && !bad) {
        tc_fence_after();
        const uint32_t base = smem_u32(sm.kq);
        constexpr uint32_t id = idesc_bf16(128, 64, false, false);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = (k / 4) * (2 * kTile) + (k % 4) * 32;
            mma_bf16(tmem, smem_desc(base + off, 16, 1024), smem_desc(base + off, 16, 1024), id,
                     k > 0);
        }
        mma_commit(&sm.mma_bar);
    }
    bad |= !mbar_wait(&sm.mma_bar, 0);
    tc_fence_after();
    if (__syncthreads_or(bad)) {
        if (tid == 0) atomicExch(err, kErrTimeout);
        goto done;
    }
    {
        // Rows of [K K^T; Q K^T]: warps 0-1 hold K K^T rows 0-63 (lanes 0-63),
        // warps 2-3 hold Q K^T rows 0-63 (lanes 64-127).
        float row[C];
        if (warp < 4) {
            uint32_t r[32];
            const uint32_t ta = tmem + ((uint32_t)(32 * warp) << 16);
            tmem_ld32(ta, r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) row[j] = __uint_as_float(r[j]);
            tmem_ld32(ta + 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) row[32 + j] = __uint_as_float(r[j]);
        }
        const int rr = (warp & 1) * 32 + lane;  // row index 0..63 within K K^T or Q K^T
        for (int j0 = 0; j0 < G; j0 += 3) {
            const int nh = min(3, G - j0);
            __syncthreads();  // previous round done with A / gam
            if (warp < nh) {
                const int h = hk * G + j0 + warp;
                chunk_gamma(g, tok0, L, Hv, h, sm.gam[warp], sm.beta[warp], beta);
            }
            __syncthreads();
            if (warp < 2) {
                // A rows (strictly lower): A_ti = b_t e^{gamma_t - gamma_i} kk_ti.
                for (int j = 0; j < nh; ++j) {
                    const float gt = sm.gam[j][rr], bt = sm.beta[j][rr];
#pragma unroll
                    for (int i = 0; i < C; ++i)
                        sm.A[j][rr][i] = i < rr ? bt * expf(gt - sm.gam[j][i]) * row[i] : 0.f;
                }
            } else if (warp < 4) {
                // P rows: P_ri = e^{gamma_r - gamma_i} qk_ri for i <= r, bf16, swizzled.
                for (int j = 0; j < nh; ++j) {
                    const int h = hk * G + j0 + j;
                    const float gr = sm.gam[j][rr];
                    uint8_t *dst = tiles + (((size_t)ch * Hv + h) * 2 + 1) * kTile;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        uint32_t w[4];
#pragma unroll
                        for (int x = 0; x < 4; ++x) {
                            const int i0 = 8 * c + 2 * x, i1 = i0 + 1;
                            const float p0 = i0 <= rr ? expf(gr - sm.gam[j][i0]) * row[i0] : 0.f;
                            const float p1 = i1 <= rr ? expf(gr - sm.gam[j][i1]) * row[i1] : 0.f;
                            w[x] = pack_bf16(p0, p1);
                        }
                        *reinterpret_cast<uint4 *>(dst + swz(rr, c)) =
                            make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
            __syncthreads();
            // T = (I + A)^-1, one column per thread, forward substitution.
            const int j = tid / C, col = tid % C;
            float tcol[C];
            if (j < nh) {
#pragma unroll
                for (int t = 0; t < C; ++t) {
                    float a0 = (t == col) ? 1.f : 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
                    const float *Arow = sm.A[j][t];
#pragma unroll
                    for (int i = 0; i < (t & ~3); i += 4) {
                        const float4 av = *reinterpret_cast<const float4 *>(Arow + i);
                        a0 = fmaf(-av.x, tcol[i], a0);
                        a1 = fmaf(-av.y, tcol[i + 1], a1);
                        a2 = fmaf(-av.z, tcol[i + 2], a2);
                        a3 = fmaf(-av.w, tcol[i + 3], a3);
                    }
#pragma unroll
                    for (int i = (t & ~3); i < t; ++i) a0 = fmaf(-Arow[i], tcol[i], a0);
                    tcol[t] = (a0 + a1) + (a2 + a3);
                }
            }
            __syncthreads();  // every column solve done reading A
            if (j < nh) {
#pragma unroll
                for (int t = 0; t < C; ++t) sm.A[j][t][col] = tcol[t];
            }
            __syncthreads();
            // T diag(b) rows -> bf16 swizzled tile.
            if (j < nh) {
                const int h = hk * G + j0 + j, t = col;
                uint8_t *dst = tiles + (((size_t)ch * Hv + h) * 2 + 0) * kTile;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const float4 x0 = *reinterpret_cast<const float4 *>(&sm.A[j][t][8 * c]);
                    const float4 x1 = *reinterpret_cast<const float4 *>(&sm.A[j][t][8 * c + 4]);
                    const float *b = &sm.beta[j][8 * c];
                    *reinterpret_cast<uint4 *>(dst + swz(t, c)) = make_uint4(
                        pack_bf16(x0.x * b[0], x0.y * b[1]), pack_bf16(x0.z * b[2], x0.w * b[3]),
                        pack_bf16(x1.x * b[4], x1.y * b[5]), pack_bf16(x1.z * b[6], x1.w * b[7]));
                }
            }
        }
    }
done:
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 64);
}

// ------------------------------------------------------------------ kernel 3
struct ChainStage {
    uint8_t k[2 * kTile];   // K tile: [64 tokens][128 dk] as two 64-column atoms
    uint8_t q[2 * kTile];
    uint8_t v[2 * kTile];
    uint8_t tb[kTile];      // T diag(b)       [64 out tokens][64 in tokens]
    uint8_t p[kTile];       // M o Q K^T       [64 out tokens][64 in tokens]
};

struct ChainSmem {
    ChainStage st[2];
    uint8_t tbg[kTile];     // T diag(b e^gamma)
    uint8_t s16[4 * kTile]; // S0 bf16, K-major: [128 dv][128 dk] as two atoms
    uint8_t wt[2 * kTile];  // W^T bf16, MN-major B operand: [128 dk rows][64 tokens]
    uint8_t dt[2 * kTile];  // Delta^T bf16: [128 dv][64 tokens]
    uint8_t dts[2 * kTile]; // Delta^T diag(e^{gamma_L - gamma})
    float gam[2][C];
    float eg[2][C];         // e^{gamma_t}
    float dec[2][C];        // e^{gamma_L - gamma_t}
    uint64_t full[2];
    uint64_t mma_bar;
    uint32_t tmem;
};

// TMEM columns
constexpr uint32_t kColU = 0, kColW = 64, kColO1 = 128, kColO2 = 192, kColS = 256;

__device__ __forceinline__ void chain_issue_loads(ChainSmem &sm, int s, const CUtensorMap *tq,
                                                  const CUtensorMap *tk, const CUtensorMap *tv,
                                                  const uint8_t *tiles, int ch, int h, int hk,
                                                  int Hv, int tok0) {
    ChainStage &st = sm.st[s];
    uint64_t *bar = &sm.full[s];
    mbar_arrive_expect_tx(bar, 8 * kTile);
    tma_load_3d(st.k, tk, 0, hk, tok0, bar);
    tma_load_3d(st.k + kTile, tk, 64, hk, tok0, bar);
    tma_load_3d(st.q, tq, 0, hk, tok0, bar);
    tma_load_3d(st.q + kTile, tq, 64, hk, tok0, bar);
    tma_load_3d(st.v, tv, 0, h, tok0, bar);
    tma_load_3d(st.v + kTile, tv, 64, h, tok0, bar);
    const uint8_t *src = tiles + ((size_t)ch * Hv + h) * 2 * kTile;
    bulk_load(st.tb, src, kTile, bar);
    bulk_load(st.p, src + kTile, kTile, bar);
}

// Loads the 64 columns [col, col + 64) of this thread's TMEM lane as floats.
__device__ __forceinline__ void tmem_row64(uint32_t taddr, float (&x)[64]) {
    uint32_t r[32];
    tmem_ld32(taddr, r);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(r[j]);
    tmem_ld32(taddr + 32, r);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 32; ++j) x[32 + j] = __uint_as_float(r[j]);
}

// Writes 64 floats as one bf16 swizzled row (128 bytes) of a K-major or
// MN-major atom column.
__device__ __forceinline__ void store_row_bf16(uint8_t *atom, int row, const float (&x)[64]) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        *reinterpret_cast<uint4 *>(atom + swz(row, c)) =
            make_uint4(pack_bf16(x[8 * c], x[8 * c + 1]), pack_bf16(x[8 * c + 2], x[8 * c + 3]),
                       pack_bf16(x[8 * c + 4], x[8 * c + 5]), pack_bf16(x[8 * c + 6], x[8 * c + 7]));
    }
}

__global__ void __launch_bounds__(kChainThreads, 1)
gdn_chain_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const float *__restrict__ g,
                 const int *__restrict__ chunk_off, const int *__restrict__ order,
                 const int4 *__restrict__ table, const uint8_t *__restrict__ tiles,
                 const float *__restrict__ h0, __nv_bfloat16 *__restrict__ out,
                 float *__restrict__ hT, int *__restrict__ err, int N, int Hk, int Hv) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    ChainSmem &sm = *reinterpret_cast<ChainSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5;
    const int n = order[blockIdx.x / Hv], h = blockIdx.x % Hv;
    const int hk = h / (Hv / Hk);
    const int c_begin = chunk_off[n], nc = chunk_off[n + 1] - c_begin;
    const size_t state_off = ((size_t)n * Hv + h) * D * D;
    const int j = tid;  // the TMEM lane / state row this thread owns
    const uint32_t lane_off = (uint32_t)(32 * warp) << 16;

    if (nc == 0) {
        // Empty sequence (or a rejected chunk table): final state = initial state.
        if (hT && !(chunk_off[N] == 0 && *err != kErrNone)) {
            for (int c = 0; c < D; c += 4) {
                float4 x = h0 ? *reinterpret_cast<const float4 *>(h0 + state_off + j * D + c)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
                *reinterpret_cast<float4 *>(hT + state_off + j * D + c) = x;
            }
        }
        return;
    }

    if (tid == 0) {
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        mbar_init(&sm.full[0], 1);
        mbar_init(&sm.full[1], 1);
        mbar_init(&sm.mma_bar, 1);
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
    const uint32_t tS = tmem + lane_off + kColS;

    int issued = 0;   // chunks whose loads have been issued
    if (tid == 0) {
        for (; issued < min(2, nc); ++issued) {
            const int4 e = table[c_begin + issued];
            chain_issue_loads(sm, issued, &tm_q, &tm_k, &tm_v, tiles, c_begin + issued, h, hk, Hv,
                              e.y);
        }
    }
    if (warp == 0) {
        const int4 e0 = table[c_begin];
        chunk_gamma(g, e0.y, e0.z, Hv, h, sm.gam[0], nullptr, nullptr, sm.eg[0], sm.dec[0]);
        if (nc > 1) {
            const int4 e1 = table[c_begin + 1];
            chunk_gamma(g, e1.y, e1.z, Hv, h, sm.gam[1], nullptr, nullptr, sm.eg[1], sm.dec[1]);
        }
    }
    __syncthreads();
    // Initial state: bf16 copy to smem, fp32 copy (pre-scaled by the first
    // chunk's total decay) to TMEM.
    {
        const float scale = expf(sm.gam[0][C - 1]);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float x[64];
#pragma unroll
            for (int c = 0; c < 64; c += 4) {
                const float4 v4 = h0 ? *reinterpret_cast<const float4 *>(
                                           h0 + state_off + (size_t)j * D + half * 64 + c)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
                x[c] = v4.x; x[c + 1] = v4.y; x[c + 2] = v4.z; x[c + 3] = v4.w;
            }
            store_row_bf16(sm.s16 + half * 2 * kTile, j, x);
            uint32_t r[32];
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {
#pragma unroll
                for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(scale * x[32 * q2 + c]);
                tmem_st32(tS + half * 64 + 32 * q2, r);
            }
        }
        tmem_st_wait();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    uint32_t mma_phase = 0;
    bool bad = false;
    const uint32_t s16 = smem_u32(sm.s16), wt = smem_u32(sm.wt), dt = smem_u32(sm.dt),
                   dts = smem_u32(sm.dts), tbg = smem_u32(sm.tbg);
    for (int c = 0; c < nc; ++c) {
        const int s = c & 1;
        ChainStage &st = sm.st[s];
        const int4 e = table[c_begin + c];
        const int tok0 = e.y, L = e.z;
        const float *eg = sm.eg[s];
        const float *dec = sm.dec[s];
        bad |= !mbar_wait(&sm.full[s], (c >> 1) & 1);
        // T diag(b e^gamma) from T diag(b): scale column i by e^{gamma_i}.
        if (tid < C) {
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
                uint4 w = *reinterpret_cast<const uint4 *>(st.tb + swz(tid, cc));
                uint32_t *wp = reinterpret_cast<uint32_t *>(&w);
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    __nv_bfloat162 b2 = *reinterpret_cast<__nv_bfloat162 *>(&wp[x]);
                    const float2 f = __bfloat1622float2(b2);
                    wp[x] = pack_bf16(f.x * eg[8 * cc + 2 * x], f.y * eg[8 * cc + 2 * x + 1]);
                }
                *reinterpret_cast<uint4 *>(sm.tbg + swz(tid, cc)) = w;
            }
        }
        fence_proxy_async_smem();
        if (__syncthreads_or(bad)) break;
        const uint32_t kt = smem_u32(st.k), qt = smem_u32(st.q), vt = smem_u32(st.v),
                       tb = smem_u32(st.tb), pt = smem_u32(st.p);
        if (tid == 0) {
            tc_fence_after();
            // U^T = V^T (T diag b)^T ; W^T = K^T (T diag(b e^gamma))^T   [M=128, N=64, K=64]
            constexpr uint32_t id = idesc_bf16(128, 64, true, false);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_bf16(tmem + kColU, smem_desc(vt + k * 2048, kTile, 1024),
                         smem_desc(tb + k * 32, 16, 1024), id, k > 0);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_bf16(tmem + kColW, smem_desc(kt + k * 2048, kTile, 1024),
                         smem_desc(tbg + k * 32, 16, 1024), id, k > 0);
            mma_commit(&sm.mma_bar);
        }
        bad |= !mbar_wait(&sm.mma_bar, mma_phase);
        mma_phase ^= 1;
        tc_fence_after();
        {
            float w[64];
            tmem_row64(tmem + lane_off + kColW, w);
            store_row_bf16(sm.wt, j, w);   // row = key dim j, 64 tokens
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(bad)) break;
        if (tid == 0) {
            tc_fence_after();
            // Delta^T = U^T - S0 W^T   [M=128 dv, N=64 tokens, K=128 dk]
            constexpr uint32_t idn = idesc_bf16(128, 64, false, true, true);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                mma_bf16(tmem + kColU, smem_desc(s16 + (k / 4) * 2 * kTile + (k % 4) * 32, 16, 1024),
                         smem_desc(wt + k * 2048, kTile, 1024), idn, 1);
            // O1^T = S0 Q^T   [M=128 dv, N=64 tokens, K=128 dk]
            constexpr uint32_t id = idesc_bf16(128, 64, false, false);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                mma_bf16(tmem + kColO1,
                         smem_desc(s16 + (k / 4) * 2 * kTile + (k % 4) * 32, 16, 1024),
                         smem_desc(qt + (k / 4) * kTile + (k % 4) * 32, 16, 1024), id, k > 0);
            mma_commit(&sm.mma_bar);
        }
        bad |= !mbar_wait(&sm.mma_bar, mma_phase);
        mma_phase ^= 1;
        tc_fence_after();
        {
            float d[64];
            tmem_row64(tmem + lane_off + kColU, d);
            store_row_bf16(sm.dt, j, d);
#pragma unroll
            for (int t = 0; t < 64; ++t) d[t] *= dec[t];
            store_row_bf16(sm.dts, j, d);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(bad)) break;
        if (tid == 0) {
            tc_fence_after();
            // O2^T = Delta^T P^T   [M=128 dv, N=64 tokens, K=64 tokens]
            constexpr uint32_t id = idesc_bf16(128, 64, false, false);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_bf16(tmem + kColO2, smem_desc(dt + k * 32, 16, 1024),
                         smem_desc(pt + k * 32, 16, 1024), id, k > 0);
            // S += (diag(e^{gamma_L - gamma}) Delta)^T K   [M=128 dv, N=128 dk, K=64 tokens]
            constexpr uint32_t ids = idesc_bf16(128, 128, false, true);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_bf16(tmem + kColS, smem_desc(dts + k * 32, 16, 1024),
                         smem_desc(kt + k * 2048, kTile, 1024), ids, 1);
            mma_commit(&sm.mma_bar);
        }
        bad |= !mbar_wait(&sm.mma_bar, mma_phase);
        mma_phase ^= 1;
        tc_fence_after();
        {
            // Output: o_t = e^{gamma_t} O1 + O2, this thread's value dim j.
            float o1[64], o2[64];
            tmem_row64(tmem + lane_off + kColO1, o1);
            tmem_row64(tmem + lane_off + kColO2, o2);
            __nv_bfloat16 *op = out + ((size_t)tok0 * Hv + h) * D + j;
            const size_t tstride = (size_t)Hv * D;
#pragma unroll
            for (int t = 0; t < 64; ++t)
                if (t < L) op[t * tstride] = __float2bfloat16_rn(fmaf(eg[t], o1[t], o2[t]));
        }
        {
            // State: bf16 copy for the next chunk and pre-scale by its decay,
            // or the final state after the last chunk.
            const bool last = (c == nc - 1);
            const float scale = last ? 1.f : expf(sm.gam[s ^ 1][C - 1]);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float x[64];
                tmem_row64(tS + half * 64, x);
                if (last) {
                    if (hT) {
                        float *dst = hT + state_off + (size_t)j * D + half * 64;
#pragma unroll
                        for (int cc = 0; cc < 64; cc += 4)
                            *reinterpret_cast<float4 *>(dst + cc) =
                                make_float4(x[cc], x[cc + 1], x[cc + 2], x[cc + 3]);
                    }
                } else {
                    store_row_bf16(sm.s16 + half * 2 * kTile, j, x);
                    uint32_t r[32];
#pragma unroll
                    for (int q2 = 0; q2 < 2; ++q2) {
#pragma unroll
                        for (int cc = 0; cc < 32; ++cc)
                            r[cc] = __float_as_uint(scale * x[32 * q2 + cc]);
                        tmem_st32(tS + half * 64 + 32 * q2, r);
                    }
                }
            }
            tmem_st_wait();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(bad)) break;
        // Stage s is free: prefetch chunk c + 2 into it.
        if (c + 2 < nc) {
            const int4 e2 = table[c_begin + c + 2];
            if (tid == 0) {
                chain_issue_loads(sm, s, &tm_q, &tm_k, &tm_v, tiles, c_begin + c + 2, h, hk, Hv,
                                  e2.y);
                ++issued;
            }
            if (warp == 1)
                chunk_gamma(g, e2.y, e2.z, Hv, h, sm.gam[s], nullptr, nullptr, sm.eg[s], sm.dec[s]);
        }
        __syncthreads();
    }
    if (bad) {
        if (tid == 0) {
            atomicExch(err, kErrTimeout);
            // Let loads still in flight land before the CTA leaves.
            for (int c = 0; c < nc && c < issued; ++c) mbar_wait(&sm.full[c & 1], (c >> 1) & 1, 100000000ll);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
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
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)C};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t prefill_tc_workspace_size(const gdn_problem &p) { return ws_layout(p).total; }

bool prefill_tc_supported(const gdn_problem &p) {
    return p.qkv_dtype == GDN_BF16 && p.head_dim_k == D && p.head_dim_v == D;
}

gdn_status launch_prefill_tc(const gdn_problem &p, const void *q, const void *k, const void *v,
                             const float *g, const float *beta, const int32_t *cu,
                             const float *h0, void *out, float *hT, cudaStream_t stream) {
    if (p.num_seqs == 0) return GDN_OK;
    const WsLayout w = ws_layout(p);
    uint8_t *ws = static_cast<uint8_t *>(p.workspace);
    int *err = reinterpret_cast<int *>(ws + w.hdr);
    int *chunk_off = reinterpret_cast<int *>(ws + w.chunk_off);
    int *order = reinterpret_cast<int *>(ws + w.order);
    int4 *table = reinterpret_cast<int4 *>(ws + w.table);
    uint8_t *tiles = ws + w.tiles;

    CUtensorMap tq, tk, tv;
    if (p.total_tokens > 0) {
        if (!encode_thd(&tq, q, p.total_tokens, p.num_k_heads) ||
            !encode_thd(&tk, k, p.total_tokens, p.num_k_heads) ||
            !encode_thd(&tv, v, p.total_tokens, p.num_v_heads))
            return GDN_ERR_CUDA;
    } else {
        memset(&tq, 0, sizeof(tq));
        memset(&tk, 0, sizeof(tk));
        memset(&tv, 0, sizeof(tv));
    }

    gdn_chunk_table_kernel<<<1, 1024, 0, stream>>>(cu, p.num_seqs, p.total_tokens, w.max_chunks,
                                                    err, chunk_off, order, table);
    if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;

    if (p.total_tokens > 0) {
        const size_t smem = sizeof(PrepSmem) + 1024;
        if (cudaFuncSetAttribute(gdn_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess)
            return GDN_ERR_CUDA;
        dim3 grid((unsigned)w.max_chunks, p.num_k_heads);
        gdn_prep_kernel<<<grid, kPrepThreads, smem, stream>>>(tq, tk, g, beta, chunk_off, table,
                                                              tiles, err, p.num_seqs,
                                                              p.num_k_heads, p.num_v_heads);
        if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
    }
    const size_t smem = sizeof(ChainSmem) + 1024;
    if (cudaFuncSetAttribute(gdn_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return GDN_ERR_CUDA;
    gdn_chain_kernel<<<(unsigned)p.num_seqs * p.num_v_heads, kChainThreads, smem, stream>>>(
        tq, tk, tv, g, chunk_off, order, table, tiles, h0, static_cast<__nv_bfloat16 *>(out), hT,
        err, p.num_seqs, p.num_k_heads, p.num_v_heads);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace gdn
