// fa_bwd_launch.cuh -- host-side launch of one backward instantiation
// (fa_bwd_kernel.cuh): the D preprocess, then the key-parallel dK/dV kernel
// and the query-parallel dQ kernel, in that order on the caller's stream.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "fa_bwd_kernel.cuh"
#include "fa_launch.cuh"

namespace fa {

// Sets a kernel's dynamic shared-memory limit once per device.
template <typename K>
inline cudaError_t set_smem_once(K kern, int bytes, unsigned long long &configured) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(__atomic_load_n(&configured, __ATOMIC_ACQUIRE) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
        __atomic_fetch_or(&configured, bit, __ATOMIC_ACQ_REL);
    }
    return cudaSuccess;
}

// The three kernels of one backward, in order on the caller's stream.
// kWin: the window instantiations (kCausal false); kCap: with a softcap.
template <int D, bool kCausal, bool kBF16, bool kWin = false, bool kCap = false>
cudaError_t launch_bwd_inst(const BwdLaunch &L) {
    using C = BwdCfg<D, kBF16>;
    static unsigned long long cfg_dq = 0ull, cfg_kv = 0ull;
    auto kdq = fa_bwd_dq_kernel<D, kCausal, kBF16, kWin, kCap>;
    auto kkv = fa_bwd_dkdv_kernel<D, kCausal, kBF16, kWin, kCap>;
    cudaError_t e = set_smem_once(kdq, static_cast<int>(C::DQ_SMEM), cfg_dq);
    if (e != cudaSuccess) return e;
    e = set_smem_once(kkv, static_cast<int>(C::KV_SMEM), cfg_kv);
    if (e != cudaSuccess) return e;
    fa_bwd_delta_kernel<D, kBF16><<<L.grid_delta, 256, 0, L.stream>>>(L.args);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    kkv<<<L.grid_kv, C::NTHREADS, C::KV_SMEM, L.stream>>>(L.q, L.k, L.v, L.dout, L.args);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    kdq<<<L.grid, C::NTHREADS, C::DQ_SMEM, L.stream>>>(L.q, L.k, L.v, L.dout, L.args);
    return cudaGetLastError();
}

}  // namespace fa
