// tc_probe.cu -- GPU test probe for the tcgen05 operand layouts the prefill
// kernels use (built and run only by tests/test_tc_layouts_gpu.py).
//
// One CTA of 128 threads computes D[M=128, N] = op(A) * op(B) with bf16
// operands staged in 128-byte-swizzled shared memory by the same helpers the
// library uses, then writes D (fp32) to global memory for the host to compare
// with a plain matmul.  Modes:
//   0: A K-major [128 x K], B K-major [N x K]                (K = 128, N = 64)
//   1: A MN-major (A^T stored [K][128]), B K-major [N x K]    (K = 64,  N = 64)
//   2: A K-major [128 x K], B MN-major (B stored [K][N])      (K = 64,  N = 128)
//   3: mode 0 with A negated, accumulated onto mode 0's result
//   4: A K-major [128 x K], B MN-major (B stored [K][N])      (K = 128, N = 64)
//   5: M = 64: A K-major [64 x K], B MN-major [K][N]          (K = 64,  N = 64);
//      all 128 TMEM lanes are dumped so the host can map rows to lanes
//   6: A from TMEM [128 x K] (packed bf16 pairs per column), B K-major [N x K]
//      (K = 128, N = 64)
//   8: as 7, issued warp-uniformly by warp 0 (elect.sync inside the asm)
//  10: group latency (issue -> commit -> wait, best of 10) of MMA groups:
//      v0 1 MMA N=64; v1 8 MMAs N=64 one accumulator; v2 8 as 2 interleaved
//      accumulators; v3 8 independent accumulators; v4 4 MMAs N=128 one
//      accumulator; v5 4 MMAs N=128 as 2 accumulators (A in TMEM throughout)
//   9: timing of 64 MMAs (A smem, B K-major, warp-uniform issue) in one
//      accumulator chain vs interleaved over several accumulators:
//      v0 N=64 x1, v1 N=64 x4, v2 N=128 x1, v3 N=128 x2, v4 N=256 x1, v5 N=64 x2
//   7: timing: 64 back-to-back MMAs of mode 0's shape (N = 64) and then of
//      N = 128; d[0..3] = cycles to issue 64 (N=64), issue+complete (N=64),
//      issue 64 (N=128), issue+complete (N=128)
// Inputs (host-provided, row-major fp32, rounded to bf16 here):
//   a: mode 0/2/3/4: [128][K];  mode 1: [K][128]  (i.e. A^T)
//   b: mode 0/1/3:   [N][K];    mode 2/4: [K][N]
#include <cuda_bf16.h>
#include <stdint.h>

#include "sm103.cuh"

using namespace gdn::ptx;

// (probe only) Warp-uniform issue: every lane of the warp executes these with the same
// operands and one elected lane issues the MMA (keeps the descriptors in
// uniform registers and the warp converged).
__device__ __forceinline__ void mma_bf16_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_bf16_ta_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}


namespace {

// Stores element (row, col) of a bf16 tile held as 64-column swizzled atoms
// of `rows` rows each (atom a covers columns 64a .. 64a + 63).
__device__ void put(uint8_t *tile, int rows, int row, int col, float x) {
    const int atom = col / 64, c = col % 64;
    uint8_t *p = tile + atom * rows * 128 + swz(row, c / 8) + (c % 8) * 2;
    *reinterpret_cast<__nv_bfloat16 *>(p) = __float2bfloat16_rn(x);
}

template <int V>
__device__ void time_groups(uint32_t a0, uint32_t b0, uint32_t tmem, uint64_t *bar, float *d,
                            int &phase) {
    // v0: 8 x N=64, A TMEM, B K-major      v1: 8 x N=64, A TMEM, B MN-major
    // v2: 8 x N=64, A smem K-major, B K-major
    // v3: 8 x N=64, A smem MN-major, B K-major
    // v4: 4 x N=128, A TMEM, B K-major     v5: 4 x N=128, A TMEM, B MN-major
    constexpr int count = V >= 4 ? 4 : 8;
    constexpr int Nn = V >= 4 ? 128 : 64;
    constexpr bool a_tm = (V == 0 || V == 1 || V == 4 || V == 5);
    constexpr bool a_mn = (V == 3);
    constexpr bool b_mn = (V == 1 || V == 5);
    const uint64_t ad = a_mn ? smem_desc(a0, 8192, 1024) : smem_desc(a0, 16, 1024);
    const uint64_t bd = b_mn ? smem_desc(b0, 8192, 1024) : smem_desc(b0, 16, 1024);
    constexpr uint32_t id = idesc_bf16(128, Nn, a_mn, b_mn);
    long long best = 1ll << 40;
    for (int rep = 0; rep < 10; ++rep) {
        const long long t0 = clock64();
#pragma unroll
        for (int r = 0; r < count; ++r) {
            const uint64_t b = b_mn ? bd + 128 * (r % 4) : bd + 2 * (r % 4);
            if (a_tm)
                mma_bf16_ta_w(tmem, tmem + 384 + 8 * (r % 8), b, id, r > 0);
            else
                mma_bf16_w(tmem, a_mn ? ad + 128 * (r % 4) : ad + 2 * (r % 4), b, id, r > 0);
        }
        mma_commit_w(bar);
        warp_wait_poll(bar, phase & 1);
        ++phase;
        const long long t1 = clock64();
        best = min(best, t1 - t0);
    }
    if ((threadIdx.x & 31) == 0) d[V] = (float)best;
}

template <int V>
__device__ void time_chains(uint32_t a0, uint32_t b0, uint32_t tmem, uint64_t *bar, float *d) {
    constexpr int Nn = (V <= 1 || V == 5) ? 64 : (V <= 3 ? 128 : 256);
    constexpr int chains = V == 1 ? 4 : (V == 3 || V == 5 ? 2 : 1);
    const uint64_t ad = smem_desc(a0, 16, 1024);
    const uint64_t bd = smem_desc(b0, 16, 1024);
    constexpr uint32_t id = idesc_bf16(128, Nn, false, false);
    const long long t0 = clock64();
#pragma unroll
    for (int r = 0; r < 64; ++r)
        mma_bf16_w(tmem + (r % chains) * Nn, ad + 2 * (r % 4), bd + 2 * (r % 4), id, r >= chains);
    const long long t1 = clock64();
    mma_commit_w(bar);
    warp_wait_poll(bar, V & 1);
    const long long t2 = clock64();
    if ((threadIdx.x & 31) == 0) {
        d[2 * V] = (float)(t1 - t0);
        d[2 * V + 1] = (float)(t2 - t0);
    }
}

template <int V>
__device__ void time_variant(int mode, uint32_t a0, uint32_t b0, uint32_t tmem, uint64_t *bar,
                             float *d) {
    constexpr int Nn = (V == 1 || V == 5) ? 128 : 64;
    constexpr bool a_tm = (V == 2 || V == 3 || V == 5);
    constexpr bool b_mn = (V == 3 || V == 4 || V == 5);
    const uint64_t ad = smem_desc(a0, 16, 1024);
    const uint64_t bd = b_mn ? smem_desc(b0, 8192, 1024) : smem_desc(b0, 16, 1024);
    constexpr uint32_t id = idesc_bf16(128, Nn, false, b_mn);
    const bool warp_mode = (mode == 8);
    const long long t0 = clock64();
#pragma unroll
    for (int r = 0; r < 64; ++r) {
        const uint64_t b = b_mn ? bd + 128 * (r % 4) : bd + 2 * (r % 4);
        if (warp_mode) {
            if (a_tm) mma_bf16_ta_w(tmem, tmem + 128 + 8 * (r % 8), b, id, r > 0);
            else mma_bf16_w(tmem, ad + 2 * (r % 4), b, id, r > 0);
        } else {
            if (a_tm) mma_bf16_ta(tmem, tmem + 128 + 8 * (r % 8), b, id, r > 0);
            else mma_bf16(tmem, ad + 2 * (r % 4), b, id, r > 0);
        }
    }
    const long long t1 = clock64();
    if (warp_mode) mma_commit_w(bar); else mma_commit(bar);
    if (warp_mode) warp_wait_poll(bar, V & 1); else mbar_wait(bar, V & 1, 2000000000ll);
    const long long t2 = clock64();
    if ((threadIdx.x & 31) == 0) {
        d[2 * V] = (float)(t1 - t0);
        d[2 * V + 1] = (float)(t2 - t0);
    }
}

}  // namespace

extern "C" __global__ void __launch_bounds__(128) tc_probe_kernel(const float *a, const float *b,
                                                                  float *d, int mode,
                                                                  int *status) {
    __shared__ __align__(1024) uint8_t sa[32768];
    __shared__ __align__(1024) uint8_t sb[32768];
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t tslot;
    const int tid = threadIdx.x, warp = tid / 32;
    const int K = (mode == 1 || mode == 2 || mode == 5) ? 64 : 128;
    const int M = (mode == 5) ? 64 : 128;
    const int N = (mode == 2) ? 128 : 64;

    if (mode == 5)
        for (int i = tid; i < 128 * 64; i += 128) d[i] = 0.f;
    // Stage operands.
    if (mode == 1) {            // A^T stored [K rows][128 M]: MN-major, atoms over M
        for (int i = tid; i < K * 128; i += 128) put(sa, K, i / 128, i % 128, a[i]);
    } else {                    // A [M rows][K]: K-major, atoms over K
        for (int i = tid; i < M * K; i += 128) put(sa, M, i / K, i % K, a[i]);
    }
    if (mode == 9 || mode == 10) {  // B [256 rows][64]: one atom of 32 KB
        for (int i = tid; i < 256 * 64; i += 128) put(sb, 256, i / 64, i % 64, b[i % (64 * 128)]);
    } else if (mode == 7) {     // B [128 rows][K] so both N = 64 and N = 128 read valid data
        for (int i = tid; i < 128 * K; i += 128) put(sb, 128, i / K, i % K, b[i % (64 * K)]);
    } else if (mode == 2 || mode == 4 || mode == 5) {  // B stored [K rows][N]: MN-major, atoms over N
        for (int i = tid; i < K * N; i += 128) put(sb, K, i / N, i % N, b[i]);
    } else {                    // B [N rows][K]: K-major
        for (int i = tid; i < N * K; i += 128) put(sb, N, i / K, i % K, b[i]);
    }
    fence_proxy_async_smem();
    if (warp == 0) {
        tmem_alloc(&tslot, mode == 10 ? 512 : 256);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tslot;
    const uint32_t a0 = smem_u32(sa), b0 = smem_u32(sb);
    if (mode == 6) {
        // A row tid into TMEM columns 128.. as packed bf16 pairs.
        for (int c0 = 0; c0 < K / 2; c0 += 32) {
            uint32_t r[32];
            for (int c = 0; c < 32; ++c)
                r[c] = pack_bf16(a[tid * K + 2 * (c0 + c)], a[tid * K + 2 * (c0 + c) + 1]);
            tmem_st32(tmem + ((uint32_t)(32 * warp) << 16) + 128 + c0, r);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    if (mode == 10) {
        if (warp == 0) {
            int phase = 0;
            time_groups<0>(a0, b0, tmem, &bar, d, phase);
            time_groups<1>(a0, b0, tmem, &bar, d, phase);
            time_groups<2>(a0, b0, tmem, &bar, d, phase);
            time_groups<3>(a0, b0, tmem, &bar, d, phase);
            time_groups<4>(a0, b0, tmem, &bar, d, phase);
            time_groups<5>(a0, b0, tmem, &bar, d, phase);
        }
        tc_fence_before();
        __syncthreads();
        if (warp == 0) tmem_dealloc(tmem, 512);
        return;
    }
    if (mode == 9) {
        if (warp == 0) {
            time_chains<0>(a0, b0, tmem, &bar, d);
            time_chains<1>(a0, b0, tmem, &bar, d);
            time_chains<2>(a0, b0, tmem, &bar, d);
            time_chains<3>(a0, b0, tmem, &bar, d);
            time_chains<4>(a0, b0, tmem, &bar, d);
            time_chains<5>(a0, b0, tmem, &bar, d);
        }
        tc_fence_before();
        __syncthreads();
        if (warp == 0) tmem_dealloc(tmem, 256);
        return;
    }
    if (mode == 7 || mode == 8) {
        // Timing of 64 back-to-back MMAs (M = 128, K = 16) per variant:
        // 0: A smem K-major, B K-major, N=64     1: same, N=128
        // 2: A TMEM,         B K-major, N=64     3: A TMEM, B MN-major, N=64
        // 4: A smem K-major, B MN-major, N=64    5: A TMEM, B MN-major, N=128
        // d[2v] = issue cycles, d[2v+1] = issue + completion cycles.
        if (mode == 7 ? tid == 0 : warp == 0) {
            time_variant<0>(mode, a0, b0, tmem, &bar, d);
            time_variant<1>(mode, a0, b0, tmem, &bar, d);
            time_variant<2>(mode, a0, b0, tmem, &bar, d);
            time_variant<3>(mode, a0, b0, tmem, &bar, d);
            time_variant<4>(mode, a0, b0, tmem, &bar, d);
            time_variant<5>(mode, a0, b0, tmem, &bar, d);
        }
        tc_fence_before();
        __syncthreads();
        if (warp == 0) tmem_dealloc(tmem, 256);
        return;
    }
    if (tid == 0) {
        const int reps = (mode == 3) ? 2 : 1;
        for (int rep = 0; rep < reps; ++rep) {
            for (int k = 0; k < K / 16; ++k) {
                uint64_t ad, bd;
                if (mode == 6) {
                    mma_bf16_ta(tmem, tmem + 128 + 8 * k,
                                smem_desc(b0 + (k / 4) * (N * 128) + (k % 4) * 32, 16, 1024),
                                idesc_bf16(128, N, false, false), k > 0);
                    continue;
                }
                if (mode == 1)
                    ad = smem_desc(a0 + k * 2048, K * 128, 1024);
                else
                    ad = smem_desc(a0 + (k / 4) * (M * 128) + (k % 4) * 32, 16, 1024);
                if (mode == 2 || mode == 4 || mode == 5)
                    bd = smem_desc(b0 + k * 2048, K * 128, 1024);
                else
                    bd = smem_desc(b0 + (k / 4) * (N * 128) + (k % 4) * 32, 16, 1024);
                const uint32_t id = idesc_bf16(M, N, mode == 1, mode == 2 || mode == 4 || mode == 5,
                                               rep == 1);
                mma_bf16(tmem, ad, bd, id, (k > 0 || rep > 0) ? 1u : 0u);
            }
        }
        mma_commit(&bar);
    }
    const bool ok = mbar_wait(&bar, 0, 2000000000ll);
    tc_fence_after();
    if (!ok && status) atomicExch(status, 1);
    for (int c0 = 0; c0 < N; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + c0, r);
        tmem_ld_wait();
        for (int j = 0; j < 32; ++j) d[tid * N + c0 + j] = __uint_as_float(r[j]);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

extern "C" int tc_probe_run(const float *a, const float *b, float *d, int mode, int *status) {
    tc_probe_kernel<<<1, 128>>>(a, b, d, mode, status);
    if (cudaGetLastError() != cudaSuccess) return 1;
    return cudaDeviceSynchronize() == cudaSuccess ? 0 : 2;
}
