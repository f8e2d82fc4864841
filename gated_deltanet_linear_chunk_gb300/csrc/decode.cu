// decode.cu -- single-token recurrent step of the Gated DeltaNet layer.
//
// Per (sequence n, value head h), with a = exp(g), b = beta and the updated
// state used for the output (the recurrence S_t = a S_{t-1} (I - b k k^T) +
// b v k^T, o_t = S_t q; Gated DeltaNet layers of the hybrid Qwen3.8-27B model,
// page "reactapp.top", section "Exploiter l'architecture hybride": a
// fixed-size fp32 state per conversation):
//
//   x = S k,  y = S q                       (one pass over each state row)
//   delta = b (v - a x)
//   S <- a S + delta k^T                    (in place)
//   o = S_new q = a y + (k . q) delta
//
// The state may also be stored in 16 bits (fp16 or bf16; the same page
// reports the fork keeping it in fp16 at unchanged perplexity): it is then
// read, updated in fp32 and stored rounded to nearest even.
//
// The step is a read-modify-write of the state, so it is bound by HBM
// bandwidth: 2 * dv * dk * sizeof(state) bytes per (n, h) against ~6 dv dk
// flops.  Each warp owns whole state rows: lane l holds dk/32 consecutive
// elements of a row (16-byte loads for an fp32 state with dk = 128, 8-byte
// loads for a 16-bit one), the two dot products are warp-shuffle reductions,
// and kDecodeRows rows are loaded before any is reduced so that every lane
// keeps several loads in flight; the next batch of rows is loaded while the
// current one is reduced and stored.  Loads and stores carry the streaming
// (evict-first) hint: the state is touched once per step.
#include <cuda_fp16.h>

#include "common.cuh"

namespace gdn {
namespace {

constexpr int kDecodeWarps = 4;
constexpr int kDecodeRows = 8;  // rows per warp per iteration (also best for 16-bit states)

// EPT consecutive state elements of one lane: loaded as raw words
// (streaming loads; a 16-bit state stays packed in registers until used),
// unpacked to fp32 where needed, and stored from fp32 (streaming stores,
// round to nearest even for 16 bits).
template <typename TS, int EPT> struct StateIO;
template <> struct StateIO<float, 4> {
    using Raw = float4;
    __device__ static Raw load(const float *p) { return __ldcs(reinterpret_cast<const float4 *>(p)); }
    __device__ static void unpack(const Raw &t, float (&r)[4]) {
        r[0] = t.x; r[1] = t.y; r[2] = t.z; r[3] = t.w;
    }
    __device__ static void store(float *p, const float (&r)[4]) {
        __stcs(reinterpret_cast<float4 *>(p), make_float4(r[0], r[1], r[2], r[3]));
    }
};
template <> struct StateIO<float, 2> {
    using Raw = float2;
    __device__ static Raw load(const float *p) { return __ldcs(reinterpret_cast<const float2 *>(p)); }
    __device__ static void unpack(const Raw &t, float (&r)[2]) { r[0] = t.x; r[1] = t.y; }
    __device__ static void store(float *p, const float (&r)[2]) {
        __stcs(reinterpret_cast<float2 *>(p), make_float2(r[0], r[1]));
    }
};

// Two 16-bit values in one word, to and from fp32 (round to nearest even).
__device__ __forceinline__ float2 unpack2(uint32_t w, __half) {
    return __half22float2(*reinterpret_cast<const __half2 *>(&w));
}
__device__ __forceinline__ float2 unpack2(uint32_t w, __nv_bfloat16) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w));
}
__device__ __forceinline__ uint32_t pack2(float a, float b, __half) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}
__device__ __forceinline__ uint32_t pack2(float a, float b, __nv_bfloat16) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

template <typename TS> struct StateIO<TS, 4> {
    using Raw = uint2;
    __device__ static Raw load(const TS *p) { return __ldcs(reinterpret_cast<const uint2 *>(p)); }
    __device__ static void unpack(const Raw &t, float (&r)[4]) {
        const float2 a = unpack2(t.x, TS()), b = unpack2(t.y, TS());
        r[0] = a.x; r[1] = a.y; r[2] = b.x; r[3] = b.y;
    }
    __device__ static void store(TS *p, const float (&r)[4]) {
        __stcs(reinterpret_cast<uint2 *>(p),
               make_uint2(pack2(r[0], r[1], TS()), pack2(r[2], r[3], TS())));
    }
};
template <typename TS> struct StateIO<TS, 2> {
    using Raw = unsigned int;
    __device__ static Raw load(const TS *p) {
        return __ldcs(reinterpret_cast<const unsigned int *>(p));
    }
    __device__ static void unpack(const Raw &t, float (&r)[2]) {
        const float2 a = unpack2(t, TS());
        r[0] = a.x; r[1] = a.y;
    }
    __device__ static void store(TS *p, const float (&r)[2]) {
        __stcs(reinterpret_cast<unsigned int *>(p), pack2(r[0], r[1], TS()));
    }
};

template <typename TIn, typename TS, int DK>
__global__ void __launch_bounds__(kDecodeWarps * 32)
gdn_decode_kernel(const TIn *__restrict__ q, const TIn *__restrict__ k,
                  const TIn *__restrict__ v, const float *__restrict__ g,
                  const float *__restrict__ beta, TS *__restrict__ state,
                  TIn *__restrict__ out, int Hk, int Hv, int DV) {
    constexpr int EPT = DK / 32;
    const int nh = blockIdx.x;            // n * Hv + h
    const int n = nh / Hv, h = nh - n * Hv;
    const int hk = h / (Hv / Hk);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    float kr[EPT], qr[EPT];
    const size_t kq_off = ((size_t)n * Hk + hk) * DK + lane * EPT;
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
        kr[e] = to_f32(k[kq_off + e]);
        qr[e] = to_f32(q[kq_off + e]);
    }
    float kq = 0.f;
#pragma unroll
    for (int e = 0; e < EPT; ++e) kq = fmaf(kr[e], qr[e], kq);
    kq = warp_sum(kq);

    const float a = expf(g[nh]);
    const float b = beta[nh];
    TS *S = state + (size_t)nh * DV * DK;
    const TIn *vrow = v + (size_t)nh * DV;
    TIn *orow = out + (size_t)nh * DV;

    // Rows in batches of kDecodeRows per warp; the next batch is loaded
    // before this one is reduced, updated and stored, so its loads are in
    // flight meanwhile (the two batches are disjoint rows).
    using IO = StateIO<TS, EPT>;
    constexpr int kStep = kDecodeWarps * kDecodeRows;
    typename IO::Raw raw[kDecodeRows], nxt[kDecodeRows];
    if (warp * kDecodeRows < DV) {
#pragma unroll
        for (int r = 0; r < kDecodeRows; ++r)
            nxt[r] = IO::load(S + (size_t)(warp * kDecodeRows + r) * DK + lane * EPT);
    }
    for (int r0 = warp * kDecodeRows; r0 < DV; r0 += kStep) {
#pragma unroll
        for (int r = 0; r < kDecodeRows; ++r) raw[r] = nxt[r];
        if (r0 + kStep < DV) {
#pragma unroll
            for (int r = 0; r < kDecodeRows; ++r)
                nxt[r] = IO::load(S + (size_t)(r0 + kStep + r) * DK + lane * EPT);
        }
        float vr = lane < kDecodeRows ? to_f32(vrow[r0 + lane]) : 0.f;
        float x[kDecodeRows], y[kDecodeRows];
#pragma unroll
        for (int r = 0; r < kDecodeRows; ++r) {
            float sv[EPT];
            IO::unpack(raw[r], sv);
            float xs = 0.f, ys = 0.f;
#pragma unroll
            for (int e = 0; e < EPT; ++e) {
                xs = fmaf(sv[e], kr[e], xs);
                ys = fmaf(sv[e], qr[e], ys);
            }
            x[r] = xs;
            y[r] = ys;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
            for (int r = 0; r < kDecodeRows; ++r) {
                x[r] += __shfl_xor_sync(0xffffffffu, x[r], o);
                y[r] += __shfl_xor_sync(0xffffffffu, y[r], o);
            }
        }
        float o_mine = 0.f;
#pragma unroll
        for (int r = 0; r < kDecodeRows; ++r) {
            const float vv = __shfl_sync(0xffffffffu, vr, r);
            const float delta = b * (vv - a * x[r]);
            float sv[EPT];
            IO::unpack(raw[r], sv);
#pragma unroll
            for (int e = 0; e < EPT; ++e) sv[e] = fmaf(a, sv[e], delta * kr[e]);
            IO::store(S + (size_t)(r0 + r) * DK + lane * EPT, sv);
            const float o = fmaf(a, y[r], kq * delta);
            if (lane == r) o_mine = o;
        }
        if (lane < kDecodeRows) orow[r0 + lane] = from_f32<TIn>(o_mine);
    }
}

// Verify step of speculative decoding: K <= kMaxVerify consecutive tokens of
// each sequence from one stored state, every position's output, and the
// state after every position in its own slot (the caller keeps the slot of
// the last accepted token).  Page "reactapp.top": the target model checks a
// block of draft tokens in one pass and keeps the correct prefix (section
// "DFlash2 : rediger sept tokens en une seule passe"), with eight
// speculative state slots per request (section "Pourquoi la limite est de
// 131 072 et non de 136 429").  A warp's rows stay in fp32 registers across
// the K tokens; each slot is written in the storage type.
constexpr int kMaxVerify = 8;

template <typename TIn, typename TS, int DK>
__global__ void __launch_bounds__(kDecodeWarps * 32)
gdn_verify_kernel(const TIn *__restrict__ q, const TIn *__restrict__ k,
                  const TIn *__restrict__ v, const float *__restrict__ g,
                  const float *__restrict__ beta, const TS *__restrict__ state,
                  TS *__restrict__ slots, TIn *__restrict__ out, int Hk, int Hv, int DV, int K) {
    constexpr int EPT = DK / 32;
    __shared__ float sk[kMaxVerify][DK], sq[kMaxVerify][DK];
    __shared__ float sa[kMaxVerify], sb[kMaxVerify], skq[kMaxVerify];
    const int nh = blockIdx.x;  // n * Hv + h
    const int n = nh / Hv, h = nh - n * Hv;
    const int hk = h / (Hv / Hk);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const size_t t0 = (size_t)n * K;  // first token of the sequence

    for (int i = threadIdx.x; i < K * DK; i += kDecodeWarps * 32) {
        const int j = i / DK, e = i - j * DK;
        const size_t off = ((t0 + j) * Hk + hk) * DK + e;
        sk[j][e] = to_f32(k[off]);
        sq[j][e] = to_f32(q[off]);
    }
    __syncthreads();
    for (int j = warp; j < K; j += kDecodeWarps) {
        float kq = 0.f;
#pragma unroll
        for (int e = 0; e < EPT; ++e) kq = fmaf(sk[j][lane * EPT + e], sq[j][lane * EPT + e], kq);
        kq = warp_sum(kq);
        if (lane == 0) {
            skq[j] = kq;
            sa[j] = expf(g[(t0 + j) * Hv + h]);
            sb[j] = beta[(t0 + j) * Hv + h];
        }
    }
    __syncthreads();

    using IO = StateIO<TS, EPT>;
    const TS *S = state + (size_t)nh * DV * DK;
    for (int r0 = warp * kDecodeRows; r0 < DV; r0 += kDecodeWarps * kDecodeRows) {
        float s[kDecodeRows][EPT];
        {
            typename IO::Raw raw[kDecodeRows];
#pragma unroll
            for (int r = 0; r < kDecodeRows; ++r)
                raw[r] = IO::load(S + (size_t)(r0 + r) * DK + lane * EPT);
#pragma unroll
            for (int r = 0; r < kDecodeRows; ++r) IO::unpack(raw[r], s[r]);
        }
        for (int j = 0; j < K; ++j) {
            float kr[EPT], qr[EPT];
#pragma unroll
            for (int e = 0; e < EPT; ++e) {
                kr[e] = sk[j][lane * EPT + e];
                qr[e] = sq[j][lane * EPT + e];
            }
            const size_t tok = t0 + j;
            const float vr = lane < kDecodeRows ? to_f32(v[(tok * Hv + h) * DV + r0 + lane]) : 0.f;
            float x[kDecodeRows], y[kDecodeRows];
#pragma unroll
            for (int r = 0; r < kDecodeRows; ++r) {
                float xs = 0.f, ys = 0.f;
#pragma unroll
                for (int e = 0; e < EPT; ++e) {
                    xs = fmaf(s[r][e], kr[e], xs);
                    ys = fmaf(s[r][e], qr[e], ys);
                }
                x[r] = xs;
                y[r] = ys;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
                for (int r = 0; r < kDecodeRows; ++r) {
                    x[r] += __shfl_xor_sync(0xffffffffu, x[r], o);
                    y[r] += __shfl_xor_sync(0xffffffffu, y[r], o);
                }
            }
            const float a = sa[j], b = sb[j], kq = skq[j];
            TS *slot = slots + (tok * Hv + h) * (size_t)DV * DK;
            float o_mine = 0.f;
#pragma unroll
            for (int r = 0; r < kDecodeRows; ++r) {
                const float vv = __shfl_sync(0xffffffffu, vr, r);
                const float delta = b * (vv - a * x[r]);
#pragma unroll
                for (int e = 0; e < EPT; ++e) s[r][e] = fmaf(a, s[r][e], delta * kr[e]);
                IO::store(slot + (size_t)(r0 + r) * DK + lane * EPT, s[r]);
                const float o = fmaf(a, y[r], kq * delta);
                if (lane == r) o_mine = o;
            }
            if (lane < kDecodeRows) out[(tok * Hv + h) * DV + r0 + lane] = from_f32<TIn>(o_mine);
        }
    }
}

template <typename TIn, typename TS, int DK>
gdn_status launch_verify_typed(const gdn_problem &p, int K, const void *q, const void *k,
                               const void *v, const float *g, const float *beta,
                               const void *state, void *slots, void *out, cudaStream_t stream) {
    const unsigned blocks = (unsigned)p.num_seqs * (unsigned)p.num_v_heads;
    gdn_verify_kernel<TIn, TS, DK><<<blocks, kDecodeWarps * 32, 0, stream>>>(
        static_cast<const TIn *>(q), static_cast<const TIn *>(k), static_cast<const TIn *>(v), g,
        beta, static_cast<const TS *>(state), static_cast<TS *>(slots), static_cast<TIn *>(out),
        p.num_k_heads, p.num_v_heads, p.head_dim_v, K);
    return launch_status();
}

template <typename TS>
gdn_status launch_verify_state(const gdn_problem &p, int K, const void *q, const void *k,
                               const void *v, const float *g, const float *beta,
                               const void *state, void *slots, void *out, cudaStream_t stream) {
    const bool bf = p.qkv_dtype == GDN_BF16;
    if (p.head_dim_k == 128)
        return bf ? launch_verify_typed<__nv_bfloat16, TS, 128>(p, K, q, k, v, g, beta, state,
                                                                slots, out, stream)
                  : launch_verify_typed<float, TS, 128>(p, K, q, k, v, g, beta, state, slots,
                                                        out, stream);
    return bf ? launch_verify_typed<__nv_bfloat16, TS, 64>(p, K, q, k, v, g, beta, state, slots,
                                                           out, stream)
              : launch_verify_typed<float, TS, 64>(p, K, q, k, v, g, beta, state, slots, out,
                                                   stream);
}

template <typename TIn, typename TS, int DK>
gdn_status launch_typed(const gdn_problem &p, const void *q, const void *k, const void *v,
                        const float *g, const float *beta, void *state, void *out,
                        cudaStream_t stream) {
    const unsigned blocks = (unsigned)p.num_seqs * (unsigned)p.num_v_heads;
    gdn_decode_kernel<TIn, TS, DK><<<blocks, kDecodeWarps * 32, 0, stream>>>(
        static_cast<const TIn *>(q), static_cast<const TIn *>(k), static_cast<const TIn *>(v), g,
        beta, static_cast<TS *>(state), static_cast<TIn *>(out), p.num_k_heads, p.num_v_heads,
        p.head_dim_v);
    return launch_status();
}

template <typename TS>
gdn_status launch_state(const gdn_problem &p, const void *q, const void *k, const void *v,
                        const float *g, const float *beta, void *state, void *out,
                        cudaStream_t stream) {
    const bool bf = p.qkv_dtype == GDN_BF16;
    if (p.head_dim_k == 128)
        return bf ? launch_typed<__nv_bfloat16, TS, 128>(p, q, k, v, g, beta, state, out, stream)
                  : launch_typed<float, TS, 128>(p, q, k, v, g, beta, state, out, stream);
    return bf ? launch_typed<__nv_bfloat16, TS, 64>(p, q, k, v, g, beta, state, out, stream)
              : launch_typed<float, TS, 64>(p, q, k, v, g, beta, state, out, stream);
}

}  // namespace

gdn_status launch_verify(const gdn_problem &p, int num_tokens, const void *q, const void *k,
                         const void *v, const float *g, const float *beta, const void *state,
                         int state_dtype, void *slots, void *out, cudaStream_t stream) {
    if (p.num_seqs == 0) return GDN_OK;
    if (num_tokens < 1 || num_tokens > kMaxVerify) return GDN_ERR_INVALID_ARG;
    switch (state_dtype) {
        case GDN_F32:
            return launch_verify_state<float>(p, num_tokens, q, k, v, g, beta, state, slots, out,
                                              stream);
        case GDN_F16:
            return launch_verify_state<__half>(p, num_tokens, q, k, v, g, beta, state, slots,
                                               out, stream);
        case GDN_BF16:
            return launch_verify_state<__nv_bfloat16>(p, num_tokens, q, k, v, g, beta, state,
                                                      slots, out, stream);
    }
    return GDN_ERR_UNSUPPORTED;
}

gdn_status launch_decode(const gdn_problem &p, const void *q, const void *k, const void *v,
                         const float *g, const float *beta, void *state, int state_dtype,
                         void *out, cudaStream_t stream) {
    if (p.num_seqs == 0) return GDN_OK;
    switch (state_dtype) {
        case GDN_F32: return launch_state<float>(p, q, k, v, g, beta, state, out, stream);
        case GDN_F16: return launch_state<__half>(p, q, k, v, g, beta, state, out, stream);
        case GDN_BF16:
            return launch_state<__nv_bfloat16>(p, q, k, v, g, beta, state, out, stream);
    }
    return GDN_ERR_UNSUPPORTED;
}

}  // namespace gdn
