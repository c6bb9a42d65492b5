// fa_launch.cuh -- host-side launch record shared by the C-ABI translation
// unit (fa_api.cu) and the per-head-dim kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "fa_bwd_kernel.cuh"
#include "fa_fwd_1q_kernel.cuh"
#include "fa_fwd_fp8_1q_kernel.cuh"
#include "fa_fwd_kernel.cuh"

namespace fa {

struct FwdLaunch {
    CUtensorMap q, k, v;   // 4-D maps {d, H, N, B}, box {64, 1, 128, 1}, 128-B swizzle
    FwdArgs args;
    int grid;              // persistent CTAs (<= SM count)
    cudaStream_t stream;
    bool causal;
    bool bf16;
    bool d64;              // split and variant paths: head dim 64 (else 128)
};

cudaError_t launch_fwd_d64(const FwdLaunch &L);
cudaError_t launch_fwd_d128(const FwdLaunch &L);
cudaError_t launch_fwd_d256(const FwdLaunch &L);   // K/V maps with 64-row boxes
cudaError_t launch_fwd_fp8(const FwdLaunch &L);    // e4m3 maps, 128-byte boxes
cudaError_t launch_fwd_fp8_d256(const FwdLaunch &L);   // the same at head dim 256
cudaError_t launch_fwd_split(const FwdLaunch &L);  // split key ranges, d in {64, 128}
cudaError_t launch_fwd_ext(const FwdLaunch &L);    // window / sinks, d in {64, 128}
cudaError_t launch_fwd_ext_softcap(const FwdLaunch &L);   // the same with a softcap
// Grouped heads packed into the Q tiles (q map box {64, group, 128 / group, 1}),
// d in {64, 128}, plain or causal.
cudaError_t launch_fwd_pack(const FwdLaunch &L);
// Split-KV combine: O, LSE from S partials (o_part [S][B][N][H][d] FP32,
// lse_part [S][B][H][N]); d in {64, 128}.
struct CombineArgs {
    const float *o_part, *lse_part;
    void *o;
    float *lse;
    int B, H, N, d, S, n_kv, causal;
    bool bf16;
};
cudaError_t launch_combine(const CombineArgs &a, int grid, cudaStream_t stream);

// Backward: maps {d, H, N, B} with box {64, 1, 128, 1} (128-byte swizzle)
// for Q, K, V and dO; grid = persistent CTAs of both main kernels.
struct BwdLaunch {
    CUtensorMap q, k, v, dout;
    BwdArgs args;
    int grid;              // dQ kernel
    int grid_kv;           // dK/dV kernel (units over K/V heads)
    int grid_delta;
    int d;
    bool causal;
    bool bf16;
    cudaStream_t stream;
};
cudaError_t launch_bwd(const BwdLaunch &L);
// The same for a local window (L.args.wl, L.args.wr; L.causal unused).
cudaError_t launch_bwd_win(const BwdLaunch &L);
// Failure-path self-test: bounded waits that run out (fa_selftest.cu).
cudaError_t launch_selftest_timeout(uint32_t *status, uint32_t *result, cudaStream_t stream);
// The same with a softcap (L.args.sc_pre, L.args.sc_post).
cudaError_t launch_bwd_win_softcap(const BwdLaunch &L);
// Gradient of per-head sink logits: dsinks[h] = -sum_{b,i} 2^(sigma_h log2 e
// - LSE2_i) D_i over the workspace rows of the backward (one CTA per head).
cudaError_t launch_bwd_dsink(const BwdArgs &a, const float *sinks, float *dsinks,
                             cudaStream_t stream);

// FP8 pre-pass: persistent CTAs over (b, h, 128-row tile); x arrives by
// TMA (map {d, H, N, B}, box {d, 1, 128, 1}, no swizzle, rows >= N zero).
struct QuantArgs {
    uint8_t *x8;            // e4m3 codes, [B][N][H][d]
    float *scales;          // [B][H][n_tiles]
    const float *signs;     // +-1 diagonal of the rotation, or null
    const float *scale_in;  // given per-tile scales (kGiven pass), else unused
    uint32_t *status;       // device status word
    int B, H, N, n_tiles, total;   // total = B * H * n_tiles
};
struct QuantLaunch {
    CUtensorMap x;
    CUtensorMap x8;         // rotated pass: codes {d, H, N, B}, box {128, 1, 128, 1}, 128-B swizzle
    QuantArgs args;
    int d;
    int sm_count;
    int granularity;        // 0 per 128-row tile, 1 per head, 2 per tensor
    cudaStream_t stream;
};
cudaError_t launch_quantize(const QuantLaunch &L);

// Shared helper: set the dynamic shared-memory limit once per device, then
// launch one instantiation.
template <int D, bool kCausal, bool kBF16, bool kFP8 = false, bool kSplit = false,
          int kVar = 0, bool kPack = false>
cudaError_t launch_fwd_inst(const FwdLaunch &L) {
    using Cfg = FwdCfg<D, kCausal, kBF16, kFP8>;
    auto kern = fa_fwd_kernel<D, kCausal, kBF16, kFP8, kSplit, kVar, kPack>;
    static unsigned long long configured = 0ull;   // bit per device id (< 64)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(__atomic_load_n(&configured, __ATOMIC_ACQUIRE) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(Cfg::SMEM_BYTES));
        if (e != cudaSuccess) return e;
        __atomic_fetch_or(&configured, bit, __ATOMIC_ACQ_REL);
    }
    kern<<<L.grid, Cfg::NTHREADS, Cfg::SMEM_BYTES, L.stream>>>(L.q, L.k, L.v, L.args);
    return cudaGetLastError();
}

// Same, for the one-Q-tile schedule used at head dim 256.
template <int D, bool kCausal, bool kBF16>
cudaError_t launch_fwd_1q_inst(const FwdLaunch &L) {
    using Cfg = Fwd1qCfg<D, kCausal, kBF16>;
    auto kern = fa_fwd_1q_kernel<D, kCausal, kBF16>;
    static unsigned long long configured = 0ull;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(__atomic_load_n(&configured, __ATOMIC_ACQUIRE) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(Cfg::SMEM_BYTES));
        if (e != cudaSuccess) return e;
        __atomic_fetch_or(&configured, bit, __ATOMIC_ACQ_REL);
    }
    kern<<<L.grid, Cfg::NTHREADS, Cfg::SMEM_BYTES, L.stream>>>(L.q, L.k, L.v, L.args);
    return cudaGetLastError();
}

// Same, for the FP8 one-Q-tile kernel (head dim 256).
template <int D, bool kCausal>
cudaError_t launch_fwd_fp8_1q_inst(const FwdLaunch &L) {
    using Cfg = Fp8Fwd1qCfg<D, kCausal>;
    auto kern = fa_fwd_fp8_1q_kernel<D, kCausal>;
    static unsigned long long configured = 0ull;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(__atomic_load_n(&configured, __ATOMIC_ACQUIRE) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(Cfg::SMEM_BYTES));
        if (e != cudaSuccess) return e;
        __atomic_fetch_or(&configured, bit, __ATOMIC_ACQ_REL);
    }
    kern<<<L.grid, Cfg::NTHREADS, Cfg::SMEM_BYTES, L.stream>>>(L.q, L.k, L.v, L.args);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_fwd_dispatch(const FwdLaunch &L) {
    if (L.causal) {
        return L.bf16 ? launch_fwd_inst<D, true, true>(L) : launch_fwd_inst<D, true, false>(L);
    }
    return L.bf16 ? launch_fwd_inst<D, false, true>(L) : launch_fwd_inst<D, false, false>(L);
}

// Split key ranges (partials + combine), d in {64, 128}.
template <int D>
cudaError_t launch_fwd_split_dispatch(const FwdLaunch &L) {
    if (L.causal)
        return L.bf16 ? launch_fwd_inst<D, true, true, false, true>(L)
                      : launch_fwd_inst<D, true, false, false, true>(L);
    return L.bf16 ? launch_fwd_inst<D, false, true, false, true>(L)
                  : launch_fwd_inst<D, false, false, false, true>(L);
}

// Grouped heads packed into the Q tiles, d in {64, 128}.
template <int D>
cudaError_t launch_fwd_pack_dispatch(const FwdLaunch &L) {
    if (L.causal)
        return L.bf16 ? launch_fwd_inst<D, true, true, false, false, 0, true>(L)
                      : launch_fwd_inst<D, true, false, false, false, 0, true>(L);
    return L.bf16 ? launch_fwd_inst<D, false, true, false, false, 0, true>(L)
                  : launch_fwd_inst<D, false, false, false, false, 0, true>(L);
}

// Score and mask variants, d in {64, 128}: kVar 1 (window, sinks) or 2
// (window, sinks, softcap).
template <int D, int kVar>
cudaError_t launch_fwd_ext_dispatch(const FwdLaunch &L) {
    return L.bf16 ? launch_fwd_inst<D, false, true, false, false, kVar>(L)
                  : launch_fwd_inst<D, false, false, false, false, kVar>(L);
}

}  // namespace fa
