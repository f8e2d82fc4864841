// prefill_simt.cu -- chunked prefill on the FFMA pipes (fp32 check path).
//
// The chunked (WY/UT) form of the Gated DeltaNet recurrence with chunk length
// 64, split into intra-chunk prep, inter-chunk state recurrence and output as
// the page "cf-1.com" (section "三个优化", item 2 "GDN prefill") describes it.
// For a chunk of L <= 64 tokens starting from state S0 (dv x dk), with
// gamma_r = g_1 + ... + g_r:
//
//   A_ti  = b_t e^{gamma_t - gamma_i} (k_t . k_i),  i < t        (prep)
//   T     = (I + A)^-1                                           (prep)
//   W     = T diag(b e^gamma) K,   U = T diag(b) V                (prep)
//   Delta = U - W S0^T                                           (recurrence)
//   O     = diag(e^gamma) Q S0^T + (M o Q K^T) Delta,
//           M_ri = e^{gamma_r - gamma_i} for i <= r              (output)
//   S     = e^{gamma_L} S0 + sum_i e^{gamma_L - gamma_i} Delta_i k_i^T
//
// Tokens past the end of a sequence are given b = 0 and g = 0, which makes
// their rows of W, U and Delta zero and leaves gamma_L at the last real
// token, so a short last chunk needs no other special case.
//
// This kernel keeps everything in fp32 and is the path for fp32 inputs.  One
// CTA owns one (sequence, value head, 32-wide slice of dv) and walks the
// sequence's chunks in order, so the state slice stays in shared memory for
// the whole sequence.  The prep (K K^T, the triangular solve, W) is repeated
// by the dv / 32 slices of a head; this path is about exactness, not speed.
#include "common.cuh"

namespace gdn {
namespace {

constexpr int C = 64;        // chunk length
constexpr int SL = 32;       // dv columns per CTA
constexpr int kThreads = 256;

template <int DK> struct SimtSmem {
    float K[C][DK + 1];
    float Q[C][DK + 1];
    float W[C][DK + 1];
    float S[SL][DK + 1];     // state slice: rows = value dims, cols = key dims
    float A[C][C + 1];
    float T[C][C + 1];
    float P[C][C + 1];       // M o Q K^T
    float V[C][SL + 1];
    float D[C][SL + 1];      // U, then Delta
    float gam[C];            // inclusive cumsum of g
    float eg[C];             // e^{gamma}
    float dec[C];            // e^{gamma_L - gamma}
    float beta[C];
};

template <typename TIn, int DK>
__global__ void __launch_bounds__(kThreads, 1)
gdn_prefill_simt_kernel(const TIn *__restrict__ q, const TIn *__restrict__ k,
                        const TIn *__restrict__ v, const float *__restrict__ g,
                        const float *__restrict__ beta, const int32_t *__restrict__ cu,
                        const float *__restrict__ h0, TIn *__restrict__ out,
                        float *__restrict__ hT, int Hk, int Hv) {
    constexpr int DV = DK;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SimtSmem<DK> &sm = *reinterpret_cast<SimtSmem<DK> *>(smem_raw);
    const int tid = threadIdx.x;
    const int slice = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int hk = h / (Hv / Hk);
    const int c0 = slice * SL;
    const size_t state_off = ((size_t)n * Hv + h) * DV * DK;

    for (int idx = tid; idx < SL * DK; idx += kThreads) {
        const int r = idx / DK, c = idx - r * DK;
        sm.S[r][c] = h0 ? h0[state_off + (size_t)(c0 + r) * DK + c] : 0.f;
    }

    const int seq_begin = cu[n], seq_end = cu[n + 1];
    for (int tok0 = seq_begin; tok0 < seq_end; tok0 += C) {
        const int L = min(C, seq_end - tok0);
        __syncthreads();  // previous chunk done with the tiles
        // ---- stage the chunk ----
        for (int idx = tid; idx < C * DK; idx += kThreads) {
            const int t = idx / DK, c = idx - t * DK;
            const size_t off = ((size_t)(tok0 + t) * Hk + hk) * DK + c;
            sm.K[t][c] = t < L ? to_f32(k[off]) : 0.f;
            sm.Q[t][c] = t < L ? to_f32(q[off]) : 0.f;
        }
        for (int idx = tid; idx < C * SL; idx += kThreads) {
            const int t = idx / SL, r = idx - t * SL;
            sm.V[t][r] = t < L ? to_f32(v[((size_t)(tok0 + t) * Hv + h) * DV + c0 + r]) : 0.f;
        }
        if (tid < C) {
            const bool ok = tid < L;
            sm.gam[tid] = ok ? g[(size_t)(tok0 + tid) * Hv + h] : 0.f;
            sm.beta[tid] = ok ? beta[(size_t)(tok0 + tid) * Hv + h] : 0.f;
        }
        __syncthreads();
        if (tid == 0) {
            float acc = 0.f;
            for (int t = 0; t < C; ++t) { acc += sm.gam[t]; sm.gam[t] = acc; }
        }
        __syncthreads();
        if (tid < C) {
            sm.eg[tid] = expf(sm.gam[tid]);
            sm.dec[tid] = expf(sm.gam[C - 1] - sm.gam[tid]);
        }
        // ---- A (strictly lower) and P (lower incl. diagonal), 4x4 per thread ----
        {
            const int tb = (tid >> 4) * 4, ib = (tid & 15) * 4;
            float kk[4][4] = {}, qk[4][4] = {};
            for (int c = 0; c < DK; ++c) {
                float kt[4], qt[4], ki[4];
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    kt[x] = sm.K[tb + x][c];
                    qt[x] = sm.Q[tb + x][c];
                    ki[x] = sm.K[ib + x][c];
                }
#pragma unroll
                for (int x = 0; x < 4; ++x)
#pragma unroll
                    for (int y = 0; y < 4; ++y) {
                        kk[x][y] = fmaf(kt[x], ki[y], kk[x][y]);
                        qk[x][y] = fmaf(qt[x], ki[y], qk[x][y]);
                    }
            }
            __syncthreads();  // gam ready for everyone
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int y = 0; y < 4; ++y) {
                    const int t = tb + x, i = ib + y;
                    const float d = expf(sm.gam[t] - sm.gam[i]);
                    sm.A[t][i] = i < t ? sm.beta[t] * d * kk[x][y] : 0.f;
                    sm.P[t][i] = i <= t ? d * qk[x][y] : 0.f;
                }
        }
        __syncthreads();
        // ---- T = (I + A)^-1 by forward substitution, one column per thread ----
        if (tid < C) {
            const int j = tid;
            float col[C];
#pragma unroll
            for (int t = 0; t < C; ++t) {
                float acc = (t == j) ? 1.f : 0.f;
#pragma unroll
                for (int i = 0; i < t; ++i) acc = fmaf(-sm.A[t][i], col[i], acc);
                col[t] = acc;
            }
#pragma unroll
            for (int t = 0; t < C; ++t) sm.T[t][j] = col[t];
        }
        __syncthreads();
        // ---- W = T diag(b e^gamma) K  (4 rows x DK/16 cols per thread) ----
        {
            constexpr int CW = DK / 16;
            const int tb = (tid >> 4) * 4, cb = (tid & 15) * CW;
            float acc[4][CW] = {};
            for (int i = 0; i < C; ++i) {
                const float w = sm.beta[i] * sm.eg[i];
                float tr[4], kr[CW];
#pragma unroll
                for (int x = 0; x < 4; ++x) tr[x] = sm.T[tb + x][i];
#pragma unroll
                for (int y = 0; y < CW; ++y) kr[y] = w * sm.K[i][cb + y];
#pragma unroll
                for (int x = 0; x < 4; ++x)
#pragma unroll
                    for (int y = 0; y < CW; ++y) acc[x][y] = fmaf(tr[x], kr[y], acc[x][y]);
            }
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int y = 0; y < CW; ++y) sm.W[tb + x][cb + y] = acc[x][y];
        }
        // ---- U = T diag(b) V  (4 rows x 2 cols per thread) ----
        {
            const int tb = (tid >> 4) * 4, rb = (tid & 15) * 2;
            float acc[4][2] = {};
            for (int i = 0; i < C; ++i) {
                const float w = sm.beta[i];
                float tr[4];
#pragma unroll
                for (int x = 0; x < 4; ++x) tr[x] = sm.T[tb + x][i];
                const float v0 = w * sm.V[i][rb], v1 = w * sm.V[i][rb + 1];
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    acc[x][0] = fmaf(tr[x], v0, acc[x][0]);
                    acc[x][1] = fmaf(tr[x], v1, acc[x][1]);
                }
            }
#pragma unroll
            for (int x = 0; x < 4; ++x) { sm.D[tb + x][rb] = acc[x][0]; sm.D[tb + x][rb + 1] = acc[x][1]; }
        }
        __syncthreads();
        // ---- Delta = U - W S0^T ----
        {
            const int tb = (tid >> 4) * 4, rb = (tid & 15) * 2;
            float acc[4][2] = {};
            for (int c = 0; c < DK; ++c) {
                const float s0 = sm.S[rb][c], s1 = sm.S[rb + 1][c];
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const float w = sm.W[tb + x][c];
                    acc[x][0] = fmaf(w, s0, acc[x][0]);
                    acc[x][1] = fmaf(w, s1, acc[x][1]);
                }
            }
            __syncthreads();  // everyone has read U
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                sm.D[tb + x][rb] -= acc[x][0];
                sm.D[tb + x][rb + 1] -= acc[x][1];
            }
        }
        __syncthreads();
        // ---- O = diag(e^gamma) Q S0^T + P Delta ----
        {
            const int tb = (tid >> 4) * 4, rb = (tid & 15) * 2;
            float a1[4][2] = {}, a2[4][2] = {};
            for (int c = 0; c < DK; ++c) {
                const float s0 = sm.S[rb][c], s1 = sm.S[rb + 1][c];
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const float qv = sm.Q[tb + x][c];
                    a1[x][0] = fmaf(qv, s0, a1[x][0]);
                    a1[x][1] = fmaf(qv, s1, a1[x][1]);
                }
            }
            for (int i = 0; i < C; ++i) {
                const float d0 = sm.D[i][rb], d1 = sm.D[i][rb + 1];
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const float pv = sm.P[tb + x][i];
                    a2[x][0] = fmaf(pv, d0, a2[x][0]);
                    a2[x][1] = fmaf(pv, d1, a2[x][1]);
                }
            }
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const int t = tb + x;
                if (t < L) {
                    TIn *o = out + ((size_t)(tok0 + t) * Hv + h) * DV + c0 + rb;
                    o[0] = from_f32<TIn>(fmaf(sm.eg[t], a1[x][0], a2[x][0]));
                    o[1] = from_f32<TIn>(fmaf(sm.eg[t], a1[x][1], a2[x][1]));
                }
            }
        }
        __syncthreads();  // O done reading S0
        // ---- S = e^{gamma_L} S0 + sum_i dec_i Delta_i k_i^T  (2 rows x DK/16 cols) ----
        {
            constexpr int CS = DK / 16;
            const int rb = (tid >> 4) * 2, cb = (tid & 15) * CS;
            float acc[2][CS];
            const float eL = sm.eg[C - 1];
#pragma unroll
            for (int x = 0; x < 2; ++x)
#pragma unroll
                for (int y = 0; y < CS; ++y) acc[x][y] = eL * sm.S[rb + x][cb + y];
            for (int i = 0; i < C; ++i) {
                const float d0 = sm.dec[i] * sm.D[i][rb], d1 = sm.dec[i] * sm.D[i][rb + 1];
#pragma unroll
                for (int y = 0; y < CS; ++y) {
                    const float kv = sm.K[i][cb + y];
                    acc[0][y] = fmaf(d0, kv, acc[0][y]);
                    acc[1][y] = fmaf(d1, kv, acc[1][y]);
                }
            }
#pragma unroll
            for (int x = 0; x < 2; ++x)
#pragma unroll
                for (int y = 0; y < CS; ++y) sm.S[rb + x][cb + y] = acc[x][y];
        }
    }
    __syncthreads();
    if (hT) {
        for (int idx = tid; idx < SL * DK; idx += kThreads) {
            const int r = idx / DK, c = idx - r * DK;
            hT[state_off + (size_t)(c0 + r) * DK + c] = sm.S[r][c];
        }
    }
}

template <typename TIn, int DK>
gdn_status launch_typed(const gdn_problem &p, const void *q, const void *k, const void *v,
                        const float *g, const float *beta, const int32_t *cu, const float *h0,
                        void *out, float *hT, cudaStream_t stream) {
    auto kern = gdn_prefill_simt_kernel<TIn, DK>;
    const size_t smem = sizeof(SimtSmem<DK>);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return GDN_ERR_CUDA;
    dim3 grid(p.head_dim_v / SL, p.num_v_heads, p.num_seqs);
    kern<<<grid, kThreads, smem, stream>>>(
        static_cast<const TIn *>(q), static_cast<const TIn *>(k), static_cast<const TIn *>(v), g,
        beta, cu, h0, static_cast<TIn *>(out), hT, p.num_k_heads, p.num_v_heads);
    return launch_status();
}

}  // namespace

gdn_status launch_prefill_simt(const gdn_problem &p, const void *q, const void *k,
                               const void *v, const float *g, const float *beta,
                               const int32_t *cu, const float *h0, void *out, float *hT,
                               cudaStream_t stream) {
    if (p.num_seqs == 0) return GDN_OK;
    const bool bf = p.qkv_dtype == GDN_BF16;
    if (p.head_dim_k == 128)
        return bf ? launch_typed<__nv_bfloat16, 128>(p, q, k, v, g, beta, cu, h0, out, hT, stream)
                  : launch_typed<float, 128>(p, q, k, v, g, beta, cu, h0, out, hT, stream);
    return bf ? launch_typed<__nv_bfloat16, 64>(p, q, k, v, g, beta, cu, h0, out, hT, stream)
              : launch_typed<float, 64>(p, q, k, v, g, beta, cu, h0, out, hT, stream);
}

}  // namespace gdn
