// fa_selftest.cu -- a kernel whose bounded waits run out on purpose, so that
// the failure path every pipeline kernel relies on (mbar_wait giving up,
// the per-CTA abort flag, the device status word) can be exercised on a GPU
// without a fault: the barriers are valid, nobody arrives on them, and the
// waits end by their own time limit.
#include <cuda_runtime.h>

#include "fa_device.cuh"
#include "fa_launch.cuh"

namespace fa {

// One CTA, two warps; lane 0 of warp w waits on its own barrier (site
// w + 1), which expects one arrival that never comes.  Whichever wait
// reaches the time limit first records its role and site and raises the
// abort flag; the other then returns through the flag.  result[w] = 1 if
// warp w's wait returned false.
__global__ void __launch_bounds__(64, 1)
fa_selftest_timeout_kernel(uint32_t *status, uint32_t *result) {
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ uint32_t abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        abort_flag = 0u;
        mbar_init(smem_addr(&bars[0]), 1);
        mbar_init(smem_addr(&bars[1]), 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (lane == 0) {
        WaitCtx w{&abort_flag, status, kRoleSelftest};
        const bool ok = mbar_wait(smem_addr(&bars[warp]), 0u, w, 1u + warp);
        result[warp] = ok ? 0u : 1u;
    }
    __syncwarp();
}

cudaError_t launch_selftest_timeout(uint32_t *status, uint32_t *result, cudaStream_t stream) {
    fa_selftest_timeout_kernel<<<1, 64, 0, stream>>>(status, result);
    return cudaGetLastError();
}

}  // namespace fa
