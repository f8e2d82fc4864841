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
// The step is a read-modify-write of the fp32 state, so it is bound by HBM
// bandwidth: 2 * dv * dk * 4 bytes per (n, h) against ~6 dv dk flops.  Each
// warp owns whole state rows: lane l holds dk/32 consecutive elements of a
// row (16-byte loads for dk = 128), the two dot products are warp-shuffle
// reductions, and ROWS rows are loaded before any is reduced so that every
// lane keeps ROWS x 16 bytes in flight.  Loads and stores carry the
// streaming (evict-first) hint: the state is touched once per step.
#include "common.cuh"

namespace gdn {
namespace {

constexpr int kDecodeWarps = 4;
constexpr int kDecodeRows = 8;  // rows per warp per iteration

template <int EPT> struct Vec;
template <> struct Vec<4> {
    using T = float4;
    __device__ static void load(const float *p, float (&r)[4]) {
        float4 t = __ldcs(reinterpret_cast<const float4 *>(p));
        r[0] = t.x; r[1] = t.y; r[2] = t.z; r[3] = t.w;
    }
    __device__ static void store(float *p, const float (&r)[4]) {
        __stcs(reinterpret_cast<float4 *>(p), make_float4(r[0], r[1], r[2], r[3]));
    }
};
template <> struct Vec<2> {
    __device__ static void load(const float *p, float (&r)[2]) {
        float2 t = __ldcs(reinterpret_cast<const float2 *>(p));
        r[0] = t.x; r[1] = t.y;
    }
    __device__ static void store(float *p, const float (&r)[2]) {
        __stcs(reinterpret_cast<float2 *>(p), make_float2(r[0], r[1]));
    }
};

template <typename TIn, int DK>
__global__ void __launch_bounds__(kDecodeWarps * 32)
gdn_decode_kernel(const TIn *__restrict__ q, const TIn *__restrict__ k,
                  const TIn *__restrict__ v, const float *__restrict__ g,
                  const float *__restrict__ beta, float *__restrict__ state,
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
    float *S = state + (size_t)nh * DV * DK;
    const TIn *vrow = v + (size_t)nh * DV;
    TIn *orow = out + (size_t)nh * DV;

    for (int r0 = warp * kDecodeRows; r0 < DV; r0 += kDecodeWarps * kDecodeRows) {
        float s[kDecodeRows][EPT];
#pragma unroll
        for (int r = 0; r < kDecodeRows; ++r) Vec<EPT>::load(S + (size_t)(r0 + r) * DK + lane * EPT, s[r]);
        float vr = lane < kDecodeRows ? to_f32(vrow[r0 + lane]) : 0.f;
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
        float o_mine = 0.f;
#pragma unroll
        for (int r = 0; r < kDecodeRows; ++r) {
            const float vv = __shfl_sync(0xffffffffu, vr, r);
            const float delta = b * (vv - a * x[r]);
#pragma unroll
            for (int e = 0; e < EPT; ++e) s[r][e] = fmaf(a, s[r][e], delta * kr[e]);
            Vec<EPT>::store(S + (size_t)(r0 + r) * DK + lane * EPT, s[r]);
            const float o = fmaf(a, y[r], kq * delta);
            if (lane == r) o_mine = o;
        }
        if (lane < kDecodeRows) orow[r0 + lane] = from_f32<TIn>(o_mine);
    }
}

template <typename TIn, int DK>
gdn_status launch_typed(const gdn_problem &p, const void *q, const void *k, const void *v,
                        const float *g, const float *beta, float *state, void *out,
                        cudaStream_t stream) {
    const unsigned blocks = (unsigned)p.num_seqs * (unsigned)p.num_v_heads;
    gdn_decode_kernel<TIn, DK><<<blocks, kDecodeWarps * 32, 0, stream>>>(
        static_cast<const TIn *>(q), static_cast<const TIn *>(k), static_cast<const TIn *>(v), g,
        beta, state, static_cast<TIn *>(out), p.num_k_heads, p.num_v_heads, p.head_dim_v);
    return launch_status();
}

}  // namespace

gdn_status launch_decode(const gdn_problem &p, const void *q, const void *k, const void *v,
                         const float *g, const float *beta, float *state, void *out,
                         cudaStream_t stream) {
    if (p.num_seqs == 0) return GDN_OK;
    const bool bf = p.qkv_dtype == GDN_BF16;
    if (p.head_dim_k == 128)
        return bf ? launch_typed<__nv_bfloat16, 128>(p, q, k, v, g, beta, state, out, stream)
                  : launch_typed<float, 128>(p, q, k, v, g, beta, state, out, stream);
    return bf ? launch_typed<__nv_bfloat16, 64>(p, q, k, v, g, beta, state, out, stream)
              : launch_typed<float, 64>(p, q, k, v, g, beta, state, out, stream);
}

}  // namespace gdn
