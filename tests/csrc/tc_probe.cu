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

namespace {

// Stores element (row, col) of a bf16 tile held as 64-column swizzled atoms
// of `rows` rows each (atom a covers columns 64a .. 64a + 63).
__device__ void put(uint8_t *tile, int rows, int row, int col, float x) {
    const int atom = col / 64, c = col % 64;
    uint8_t *p = tile + atom * rows * 128 + swz(row, c / 8) + (c % 8) * 2;
    *reinterpret_cast<__nv_bfloat16 *>(p) = __float2bfloat16_rn(x);
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
    if (mode == 7) {            // B [128 rows][K] so both N = 64 and N = 128 read valid data
        for (int i = tid; i < 128 * K; i += 128) put(sb, 128, i / K, i % K, b[i % (64 * K)]);
    } else if (mode == 2 || mode == 4 || mode == 5) {  // B stored [K rows][N]: MN-major, atoms over N
        for (int i = tid; i < K * N; i += 128) put(sb, K, i / N, i % N, b[i]);
    } else {                    // B [N rows][K]: K-major
        for (int i = tid; i < N * K; i += 128) put(sb, N, i / K, i % K, b[i]);
    }
    fence_proxy_async_smem();
    if (warp == 0) {
        tmem_alloc(&tslot, 256);
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
    if (mode == 7) {
        if (tid == 0) {
            const uint64_t ad = smem_desc(a0, 16, 1024);
            for (int pass = 0; pass < 2; ++pass) {
                const int Nn = pass ? 128 : 64;
                const uint64_t bd = smem_desc(b0, 16, 1024);
                const long long t0 = clock64();
                for (int r = 0; r < 64; ++r)
                    mma_bf16(tmem, ad + 2 * (r % 4), bd + 2 * (r % 4), idesc_bf16(128, Nn, false, false), r > 0);
                const long long t1 = clock64();
                mma_commit(&bar);
                mbar_wait(&bar, pass, 2000000000ll);
                const long long t2 = clock64();
                d[2 * pass] = (float)(t1 - t0);
                d[2 * pass + 1] = (float)(t2 - t0);
            }
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
