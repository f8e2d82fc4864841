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
// flops.  The state is cut into tiles of whole rows (contiguous in memory);
// a persistent grid of one or two CTAs per SM walks the tiles with a
// cp.async pipeline a few tiles deep into shared memory, so that the next tiles
// (with their k, q, v, g and beta) are in flight while the current one is
// computed and the bytes in flight are bounded by shared memory, not by
// registers.  The compute reads a tile with L lanes per state row (8 for an
// fp32 state, 4 for a 16-bit one): lane l of a row holds the 16-byte chunks
// L j + l (j = 0, 1, ...), so the two dot products take log2 L shuffle levels
// and a warp store writes 16 L consecutive bytes of each of 32 / L rows.
// Odd rows are rotated by 4 chunks in shared memory so that the 8 lanes of
// one load phase hit distinct banks.
// Loads and stores carry the streaming (evict-first) hint: the state is
// touched once per step.
#include <cuda_fp16.h>

#include <mutex>

#include "common.cuh"

namespace gdn {
namespace {

constexpr int kDecodeThreads = 128;
constexpr int kVerifyRows = 64;          // state rows per verify CTA
constexpr int kMaxDevices = 64;

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

// One 16-byte chunk of a state row: CE elements, to and from fp32.
template <typename TS> struct Chunk {
    static constexpr int CE = 8;
    __device__ static void unpack(const uint4 &w, float *r) {
        const float2 a = unpack2(w.x, TS()), b = unpack2(w.y, TS()), c = unpack2(w.z, TS()),
                     d = unpack2(w.w, TS());
        r[0] = a.x; r[1] = a.y; r[2] = b.x; r[3] = b.y;
        r[4] = c.x; r[5] = c.y; r[6] = d.x; r[7] = d.y;
    }
    __device__ static uint4 pack(const float *r) {
        return make_uint4(pack2(r[0], r[1], TS()), pack2(r[2], r[3], TS()),
                          pack2(r[4], r[5], TS()), pack2(r[6], r[7], TS()));
    }
};
template <> struct Chunk<float> {
    static constexpr int CE = 4;
    __device__ static void unpack(const uint4 &w, float *r) {
        r[0] = __uint_as_float(w.x); r[1] = __uint_as_float(w.y);
        r[2] = __uint_as_float(w.z); r[3] = __uint_as_float(w.w);
    }
    __device__ static uint4 pack(const float *r) {
        return make_uint4(__float_as_uint(r[0]), __float_as_uint(r[1]), __float_as_uint(r[2]),
                          __float_as_uint(r[3]));
    }
};

// Input words (bf16 pairs or fp32) to fp32, exactly.
__device__ __forceinline__ void words_to_f32(uint32_t w, float *r, __nv_bfloat16) {
    r[0] = __uint_as_float(w << 16);
    r[1] = __uint_as_float(w & 0xffff0000u);
}
__device__ __forceinline__ void words_to_f32(uint32_t w, float *r, float) {
    r[0] = __uint_as_float(w);
}

// CE consecutive input elements in shared memory (16-byte aligned when CE
// elements fill 16 bytes or more, 8-byte aligned otherwise) to fp32.
template <typename TIn, int CE>
__device__ __forceinline__ void load_cvt(const TIn *p, float *r) {
    constexpr int kBytes = CE * (int)sizeof(TIn);
    constexpr int kPerWord = 4 / (int)sizeof(TIn);
    if constexpr (kBytes >= 16) {
#pragma unroll
        for (int w = 0; w < kBytes / 16; ++w) {
            const uint4 u = reinterpret_cast<const uint4 *>(p)[w];
            float *o = r + w * 4 * kPerWord;
            words_to_f32(u.x, o, TIn());
            words_to_f32(u.y, o + kPerWord, TIn());
            words_to_f32(u.z, o + 2 * kPerWord, TIn());
            words_to_f32(u.w, o + 3 * kPerWord, TIn());
        }
    } else {
        static_assert(kBytes == 8, "chunk of inputs");
        const uint2 u = *reinterpret_cast<const uint2 *>(p);
        words_to_f32(u.x, r, TIn());
        words_to_f32(u.y, r + kPerWord, TIn());
    }
}

// Lanes per state row: 8 for fp32 (a warp store then writes whole 128-byte
// lines of 4 rows), 4 for 16-bit states (64 bytes of 8 rows; fewer lanes per
// row keep the shuffle reductions short).
template <typename TS> constexpr int lanes_per_row() { return sizeof(TS) == 4 ? 8 : 4; }

// Geometry of a tile of ROWS whole state rows, LPR lanes per row.
template <typename TS, int DK, int ROWS> struct Tile {
    static constexpr int LPR = lanes_per_row<TS>();
    static constexpr int RPA = 32 / LPR;       // rows per warp access
    static constexpr int CE = Chunk<TS>::CE;   // elements per chunk
    static constexpr int CPR = DK / CE;        // chunks per row
    static constexpr int NCH = CPR / LPR;      // chunks of a row per lane
    static constexpr int EPL = NCH * CE;       // elements of a row per lane
    static constexpr int CHUNKS = ROWS * CPR;  // chunks per tile
    static constexpr int RPW = ROWS / 4;       // rows per warp
    static constexpr int ACC = RPW / RPA;      // accesses per warp
    static_assert(RPW % RPA == 0 && CHUNKS % kDecodeThreads == 0 && NCH >= 1, "tile shape");
    // Position in shared memory of chunk c of tile row r (odd rows rotated
    // by 4 chunks: the 8 lanes of a 16-byte load phase hit distinct banks).
    __device__ static int slot(int r, int c) { return r * CPR + (c ^ ((r & 1) << 2)); }
    // Chunk j of the lane's part cb of a row, and the column of its element e.
    __device__ static int chunk(int j, int cb) { return LPR * j + cb; }
    __device__ static int col(int j, int cb, int e) { return chunk(j, cb) * CE + e; }
    // Tile row of access i of the warp, for the lane's row-in-access rl.
    __device__ static int row(int warp, int i, int rl) { return warp * RPW + RPA * i + rl; }
};

// Decode pipeline shape per state type (measured on GB300, 64 x 48 heads of
// 128 x 128): state bytes per tile and tiles in flight per CTA, the current
// one included.  fp32: 4 x 32 KB, one CTA per SM; 16 bits: 6 x 16 KB, two
// CTAs per SM.
template <typename TS> constexpr int decode_tile_bytes() { return sizeof(TS) == 4 ? 32768 : 16384; }
template <typename TS> constexpr int decode_stages() { return sizeof(TS) == 4 ? 4 : 6; }

template <typename TS, int DK> constexpr int decode_rows() {
    return decode_tile_bytes<TS>() / (DK * (int)sizeof(TS)) < DK
               ? decode_tile_bytes<TS>() / (DK * (int)sizeof(TS))
               : DK;
}

__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(
                     __cvta_generic_to_shared(dst))),
                 "l"(__cvta_generic_to_global(src))
                 : "memory");
}
__device__ __forceinline__ void cp_async16_ef(void *dst, const void *src, uint64_t pol) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(__cvta_generic_to_global(src)), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(static_cast<uint32_t>(
                     __cvta_generic_to_shared(dst))),
                 "l"(__cvta_generic_to_global(src))
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Copies a tile (contiguous in global memory) into shared memory with 16-byte
// cp.async, row-rotated as Tile::slot says.  The rotation is applied to the
// source: a warp's destinations stay consecutive (one coalesced request per
// warp; permuted destinations split it and fetch sectors twice), and its
// sources are a permutation of the same 512 bytes.
template <typename G, typename TS>
__device__ __forceinline__ void tile_load_async(uint4 *tile, const TS *src, uint64_t pol) {
#pragma unroll 4
    for (int i = threadIdx.x; i < G::CHUNKS; i += kDecodeThreads) {
        const int r = i / G::CPR, c = i - r * G::CPR;
        cp_async16_ef(tile + i, reinterpret_cast<const uint4 *>(src) + G::slot(r, c), pol);
    }
}

// Sum over the LPR lanes of a row (butterfly: every lane gets the same bits).
template <int LPR> __device__ __forceinline__ float row_sum(float x) {
#pragma unroll
    for (int o = 1; o < LPR; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// The lane's columns of k and q (raw inputs in shared memory) in fp32.
template <typename G, typename TIn>
__device__ __forceinline__ void lane_kq(const TIn *sk, const TIn *sq, int cb, float (&kr)[G::EPL],
                                        float (&qr)[G::EPL]) {
#pragma unroll
    for (int j = 0; j < G::NCH; ++j) {
        load_cvt<TIn, G::CE>(sk + G::col(j, cb, 0), kr + j * G::CE);
        load_cvt<TIn, G::CE>(sq + G::col(j, cb, 0), qr + j * G::CE);
    }
}

// k . q from the lane's columns (every lane of the warp gets the same bits).
template <int LPR, int EPL> __device__ __forceinline__ float dot_kq(const float (&kr)[EPL],
                                                                    const float (&qr)[EPL]) {
    float kq = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) kq = fmaf(kr[e], qr[e], kq);
    return row_sum<LPR>(kq);
}

// One token's step on the lane's part of a state row (s in fp32, updated in
// place); returns the output element of the row.  Decode and verify both
// run this, so that a verify slot equals successive decode steps bit for bit.
template <int LPR, int EPL>
__device__ __forceinline__ float row_step(float (&s)[EPL], const float (&kr)[EPL],
                                          const float (&qr)[EPL], float a, float b, float kq,
                                          float vv) {
    float x = 0.f, y = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
        x = fmaf(s[e], kr[e], x);
        y = fmaf(s[e], qr[e], y);
    }
    x = row_sum<LPR>(x);
    y = row_sum<LPR>(y);
    const float delta = b * fmaf(-a, x, vv);
#pragma unroll
    for (int e = 0; e < EPL; ++e) s[e] = fmaf(a, s[e], delta * kr[e]);
    return fmaf(a, y, kq * delta);
}

template <typename G, typename TS>
__device__ __forceinline__ void tile_row_unpack(const uint4 *tile, int r, int cb,
                                                float (&s)[G::EPL]) {
#pragma unroll
    for (int j = 0; j < G::NCH; ++j) Chunk<TS>::unpack(tile[G::slot(r, G::chunk(j, cb))], s + j * G::CE);
}

template <typename G, typename TS>
__device__ __forceinline__ void row_store(TS *row, int cb, const float (&s)[G::EPL]) {
    uint4 *dst = reinterpret_cast<uint4 *>(row);
#pragma unroll
    for (int j = 0; j < G::NCH; ++j) __stcs(dst + G::chunk(j, cb), Chunk<TS>::pack(s + j * G::CE));
}

// Shared-memory stage of the decode pipeline: one tile with its inputs.
template <typename TIn, typename TS, int DK> struct DecodeStage {
    static constexpr int ROWS = decode_rows<TS, DK>();
    using G = Tile<TS, DK, ROWS>;
    uint4 tile[G::CHUNKS];
    alignas(16) TIn k[DK];
    alignas(16) TIn q[DK];
    alignas(16) TIn v[ROWS];
    alignas(16) float gb[4];  // g, beta
};

template <typename TIn, typename TS, int DK>
__global__ void __launch_bounds__(kDecodeThreads, 2)
gdn_decode_kernel(const TIn *__restrict__ q, const TIn *__restrict__ k,
                  const TIn *__restrict__ v, const float *__restrict__ g,
                  const float *__restrict__ beta, TS *__restrict__ state,
                  TIn *__restrict__ out, int Hk, int Hv, long long n_tiles) {
    using St = DecodeStage<TIn, TS, DK>;
    using G = typename St::G;
    constexpr int ROWS = St::ROWS;
    constexpr int TPH = DK / ROWS;  // tiles per head (dv = dk)
    constexpr int KCH = DK * (int)sizeof(TIn) / 16, VCH = ROWS * (int)sizeof(TIn) / 16;
    static_assert(2 * KCH + VCH + 2 <= kDecodeThreads, "one input copy per thread");
    constexpr int kStages = decode_stages<TS>();
    extern __shared__ __align__(16) unsigned char smem_raw[];
    St *stages = reinterpret_cast<St *>(smem_raw);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int cb = lane % G::LPR, rl = lane / G::LPR;  // lane part of its row, row in an access
    const uint64_t pol = evict_first_policy();

    // Copies tile t (rows [r0, r0 + ROWS) of head nh) and its inputs into a stage.
    auto issue = [&](long long t, St &st) {
        const long long nh = t / TPH;  // n * Hv + h
        const int r0 = (int)(t - nh * TPH) * ROWS;
        const long long n = nh / Hv;
        const int h = (int)(nh - n * Hv), hk = h / (Hv / Hk);
        tile_load_async<G>(st.tile, state + (nh * DK + r0) * DK, pol);
        const int i = threadIdx.x;
        if (i < KCH) {
            cp_async16(reinterpret_cast<uint4 *>(st.k) + i,
                       reinterpret_cast<const uint4 *>(k + (n * Hk + hk) * DK) + i);
        } else if (i < 2 * KCH) {
            cp_async16(reinterpret_cast<uint4 *>(st.q) + (i - KCH),
                       reinterpret_cast<const uint4 *>(q + (n * Hk + hk) * DK) + (i - KCH));
        } else if (i < 2 * KCH + VCH) {
            cp_async16(reinterpret_cast<uint4 *>(st.v) + (i - 2 * KCH),
                       reinterpret_cast<const uint4 *>(v + nh * DK + r0) + (i - 2 * KCH));
        } else if (i == 2 * KCH + VCH) {
            cp_async4(&st.gb[0], g + nh);
        } else if (i == 2 * KCH + VCH + 1) {
            cp_async4(&st.gb[1], beta + nh);
        }
    };

    // Launched as a programmatic dependent of the previous kernel of the
    // stream (often the previous decode step): this grid may be scheduled
    // while that one drains, and waits for it before touching memory.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const long long first = blockIdx.x, step = gridDim.x;
#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
        const long long t = first + s * step;
        if (t < n_tiles) issue(t, stages[s]);
        cp_async_commit();
    }
    int cur = 0;
    for (long long t = first; t < n_tiles; t += step) {
        cp_async_wait<kStages - 2>();  // this thread's copies of tile t have landed
        __syncthreads();               // everyone's; and the previous stage is free
        {
            const long long tn = t + (kStages - 1) * step;
            const int sn = cur == 0 ? kStages - 1 : cur - 1;
            if (tn < n_tiles) issue(tn, stages[sn]);
            cp_async_commit();
        }
        const St &st = stages[cur];
        const long long nh = t / TPH;
        const int r0 = (int)(t - nh * TPH) * ROWS;
        float kr[G::EPL], qr[G::EPL];
        lane_kq<G>(st.k, st.q, cb, kr, qr);
        const float kq = dot_kq<G::LPR>(kr, qr);
        const float a = expf(st.gb[0]), b = st.gb[1];
        TS *S = state + (nh * DK + r0) * DK;
        TIn *orow = out + nh * DK + r0;
#pragma unroll
        for (int i = 0; i < G::ACC; ++i) {
            const int r = G::row(warp, i, rl);
            float s[G::EPL];
            tile_row_unpack<G, TS>(st.tile, r, cb, s);
            const float o = row_step<G::LPR>(s, kr, qr, a, b, kq, to_f32(st.v[r]));
            row_store<G, TS>(S + (size_t)r * DK, cb, s);
            if (cb == 0) orow[r] = from_f32<TIn>(o);
        }
        cur = cur + 1 == kStages ? 0 : cur + 1;
    }
    cp_async_wait<0>();
}

// Verify step of speculative decoding: K <= kMaxVerify consecutive tokens of
// each sequence from one stored state, every position's output, and the
// state after every position in its own slot (the caller keeps the slot of
// the last accepted token).  Page "reactapp.top": the target model checks a
// block of draft tokens in one pass and keeps the correct prefix (section
// "DFlash2 : rediger sept tokens en une seule passe"), with eight
// speculative state slots per request (section "Pourquoi la limite est de
// 131 072 et non de 136 429").  A CTA takes kVerifyRows rows of one head:
// the tile and the K tokens' inputs are copied into shared memory once, each
// warp's rows stay in fp32 registers across the tokens (token-major, so each
// token's k and q are read from shared memory once per warp), and each slot
// is written in the storage type.
constexpr int kMaxVerify = 8;

template <typename TIn, typename TS, int DK>
__global__ void __launch_bounds__(kDecodeThreads)
gdn_verify_kernel(const TIn *__restrict__ q, const TIn *__restrict__ k,
                  const TIn *__restrict__ v, const float *__restrict__ g,
                  const float *__restrict__ beta, const TS *__restrict__ state,
                  TS *__restrict__ slots, TIn *__restrict__ out, int Hk, int Hv, int K) {
    constexpr int ROWS = kVerifyRows < DK ? kVerifyRows : DK;
    using G = Tile<TS, DK, ROWS>;
    constexpr int TPH = DK / ROWS;
    constexpr int KCH = DK * (int)sizeof(TIn) / 16, VCH = ROWS * (int)sizeof(TIn) / 16;
    __shared__ __align__(16) uint4 tile[G::CHUNKS];
    __shared__ __align__(16) TIn sk[kMaxVerify][DK], sq[kMaxVerify][DK], sv[kMaxVerify][ROWS];
    __shared__ float sg[kMaxVerify], sb[kMaxVerify], skq[kMaxVerify];
    const long long nh = blockIdx.x / TPH;  // n * Hv + h
    const int r0 = (int)(blockIdx.x - nh * TPH) * ROWS;
    const long long n = nh / Hv;
    const int h = (int)(nh - n * Hv), hk = h / (Hv / Hk);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int cb = lane % G::LPR, rl = lane / G::LPR;
    const long long t0 = n * K;  // first token of the sequence

    tile_load_async<G>(tile, state + (nh * DK + r0) * DK, evict_first_policy());
    for (int i = threadIdx.x; i < K * KCH; i += kDecodeThreads) {
        const int j = i / KCH, c = i - j * KCH;
        const long long off = ((t0 + j) * Hk + hk) * DK;
        cp_async16(reinterpret_cast<uint4 *>(sk[j]) + c, reinterpret_cast<const uint4 *>(k + off) + c);
        cp_async16(reinterpret_cast<uint4 *>(sq[j]) + c, reinterpret_cast<const uint4 *>(q + off) + c);
    }
    for (int i = threadIdx.x; i < K * VCH; i += kDecodeThreads) {
        const int j = i / VCH, c = i - j * VCH;
        cp_async16(reinterpret_cast<uint4 *>(sv[j]) + c,
                   reinterpret_cast<const uint4 *>(v + ((t0 + j) * Hv + h) * DK + r0) + c);
    }
    if (threadIdx.x < K) {
        cp_async4(&sg[threadIdx.x], g + (t0 + threadIdx.x) * Hv + h);
        cp_async4(&sb[threadIdx.x], beta + (t0 + threadIdx.x) * Hv + h);
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    for (int j = warp; j < K; j += kDecodeThreads / 32) {
        float kr[G::EPL], qr[G::EPL];
        lane_kq<G>(sk[j], sq[j], cb, kr, qr);
        const float kq = dot_kq<G::LPR>(kr, qr);
        if (lane == 0) skq[j] = kq;
    }
    __syncthreads();

    float s[G::ACC][G::EPL];
#pragma unroll
    for (int i = 0; i < G::ACC; ++i) tile_row_unpack<G, TS>(tile, G::row(warp, i, rl), cb, s[i]);
#pragma unroll 1
    for (int j = 0; j < K; ++j) {
        float kr[G::EPL], qr[G::EPL];
        lane_kq<G>(sk[j], sq[j], cb, kr, qr);
        const float a = expf(sg[j]), b = sb[j], kq = skq[j];
        const long long tok = t0 + j;
        TS *slot = slots + ((tok * Hv + h) * DK + r0) * DK;
        TIn *orow = out + (tok * Hv + h) * DK + r0;
#pragma unroll
        for (int i = 0; i < G::ACC; ++i) {
            const int r = G::row(warp, i, rl);
            const float o = row_step<G::LPR>(s[i], kr, qr, a, b, kq, to_f32(sv[j][r]));
            row_store<G, TS>(slot + (size_t)r * DK, cb, s[i]);
            if (cb == 0) orow[r] = from_f32<TIn>(o);
        }
    }
}

// CTAs of the persistent decode kernel on the current device (resident CTAs
// per SM times SMs), looked up once per device and kernel under a lock; 0
// when the lookup fails.
template <typename TIn, typename TS, int DK> int decode_grid() {
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
    constexpr size_t smem = decode_stages<TS>() * sizeof(DecodeStage<TIn, TS, DK>);
    int sms = 0, blocks = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaFuncSetAttribute(gdn_decode_kernel<TIn, TS, DK>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, gdn_decode_kernel<TIn, TS, DK>,
                                                      kDecodeThreads, smem) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    grid_of[dev] = blocks * sms;
    known[dev] = true;
    return grid_of[dev];
}

template <typename TIn, typename TS, int DK>
gdn_status launch_verify_typed(const gdn_problem &p, int K, const void *q, const void *k,
                               const void *v, const float *g, const float *beta,
                               const void *state, void *slots, void *out, cudaStream_t stream) {
    constexpr int ROWS = kVerifyRows < DK ? kVerifyRows : DK;
    const unsigned blocks = (unsigned)p.num_seqs * (unsigned)p.num_v_heads * (DK / ROWS);
    gdn_verify_kernel<TIn, TS, DK><<<blocks, kDecodeThreads, 0, stream>>>(
        static_cast<const TIn *>(q), static_cast<const TIn *>(k), static_cast<const TIn *>(v), g,
        beta, static_cast<const TS *>(state), static_cast<TS *>(slots), static_cast<TIn *>(out),
        p.num_k_heads, p.num_v_heads, K);
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
    const long long n_tiles = (long long)p.num_seqs * p.num_v_heads *
                              (DK / DecodeStage<TIn, TS, DK>::ROWS);
    const int max_grid = decode_grid<TIn, TS, DK>();
    if (max_grid <= 0) return GDN_ERR_CUDA;
    const long long grid = n_tiles < max_grid ? n_tiles : max_grid;
    constexpr size_t smem = decode_stages<TS>() * sizeof(DecodeStage<TIn, TS, DK>);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kDecodeThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, gdn_decode_kernel<TIn, TS, DK>, static_cast<const TIn *>(q),
                           static_cast<const TIn *>(k), static_cast<const TIn *>(v), g, beta,
                           static_cast<TS *>(state), static_cast<TIn *>(out), p.num_k_heads,
                           p.num_v_heads, n_tiles) != cudaSuccess) {
        cudaGetLastError();
        return GDN_ERR_CUDA;
    }
    return GDN_OK;
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
