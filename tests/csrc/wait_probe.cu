// wait_probe.cu -- GPU test probe for the bounded waits the library's kernels
// use (built and run only by tests/test_device_waits_gpu.py).  Nothing ever
// arrives on the probe's mbarrier, so every wait has to give up at its limit,
// say so, and let the kernel finish with the context intact.
//
// Modes (one CTA of two warps):
//   0: both warps: polling wait (warp_wait_poll, the prep units' wait) with
//      the given limit; it raises no abort flag
//   1: both warps: ready-flag wait (wait_ready, the recurrence's wait for a
//      prepped chunk) on a global flag that nothing sets, with the given limit
//   2: warp 0: all-lane wait (warp_wait_lean) with the limit; warp 1: ready-
//      flag wait with a limit 100 times longer, which must leave once warp 0
//      has raised the abort flag
//   3: both warps: all-lane wait (warp_wait_lean) with the given limit
//   4: as 2 with warp_wait_lean in both warps
// out[4 w + 0] = wait result of warp w (1 = completed), out[4 w + 1] = abort
// flag seen by warp w afterwards, out[4 w + 2] = cycles waited / 1024;
// out[8] is the ready flag (set to 0 here, never raised).
#include <stdint.h>

#include "sm103.cuh"

using namespace gdn::ptx;

extern "C" __global__ void __launch_bounds__(64) wait_probe_kernel(int mode, long long limit,
                                                                   int *out) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned *flag = reinterpret_cast<unsigned *>(out + 8);
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        abort_flag = 0;
        *flag = 0u;
    }
    __syncthreads();
    const long long t0 = clock64();
    bool ok;
    if (mode == 0)
        ok = warp_wait_poll(&bar, 0, limit);
    else if (mode == 1)
        ok = wait_ready(flag, &abort_flag, limit);
    else if (mode == 2)
        ok = warp == 0 ? warp_wait_lean(&bar, 0, &abort_flag, limit)
                       : wait_ready(flag, &abort_flag, 100 * limit);
    else if (mode == 3)
        ok = warp_wait_lean(&bar, 0, &abort_flag, limit);
    else
        ok = warp_wait_lean(&bar, 0, &abort_flag, warp == 0 ? limit : 100 * limit);
    const long long t1 = clock64();
    if (lane == 0) {
        out[4 * warp] = ok ? 1 : 0;
        out[4 * warp + 1] = *static_cast<volatile int *>(&abort_flag);
        out[4 * warp + 2] = (int)((t1 - t0) >> 10);
    }
}

extern "C" int wait_probe_run(int mode, long long limit, int *out) {
    wait_probe_kernel<<<1, 64>>>(mode, limit, out);
    if (cudaGetLastError() != cudaSuccess) return 1;
    return cudaDeviceSynchronize() == cudaSuccess ? 0 : 2;
}
