// fa_splitkv.cu -- the combine step of split-KV attention ("FlashAttention-3
// on Hopper", ch. 10: split-KV with its combine kernel; the merge is the
// block-combine rule of sec. 3.2.1 applied to finished partials):
//   LSE = log sum_s exp(LSE_s),  O = sum_s exp(LSE_s - LSE) O_s,
// where split s produced O_s (normalised over its own keys) and LSE_s.
// Memory-bound: reads S x (D + 1) FP32 values per row, writes D 16-bit
// values and one FP32.  One warp per (b, n, h) row; lane l holds elements
// [l*E, l*E + E) of the row (E = D/32).  A split whose key range holds no
// key tile of the row's query tile produced no partial and is skipped: the
// ranges are recomputed exactly as the forward kernel's work units define
// them (the pair of query tiles 2p, 2p+1 shares one key range, cut into S
// parts).
#include <cuda_runtime.h>

#include <cstdint>

#include "fa_launch.cuh"

namespace fa {

template <int D, bool kBF16>
__global__ void __launch_bounds__(256)
fa_combine_kernel(const CombineArgs a) {
    constexpr int E = D / 32;
    const long n_rows = static_cast<long>(a.B) * a.N * a.H;
    const int lane = threadIdx.x & 31;
    const long warp_g = (static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long n_warps = (static_cast<long>(gridDim.x) * blockDim.x) >> 5;
    for (long row = warp_g; row < n_rows; row += n_warps) {
        const int h = static_cast<int>(row % a.H);
        const long bn = row / a.H;
        const int n = static_cast<int>(bn % a.N), b = static_cast<int>(bn / a.N);
        // the key range of this row's query tile and of its pair
        const int m = n / 128, p = m / 2;
        auto tile_hi = [&](int mt) {
            if (mt * 128 >= a.N) return 0;
            return a.causal ? min(a.n_kv, mt + 1) : a.n_kv;
        };
        const int hi_m = tile_hi(m);
        const int Tf = max(tile_hi(2 * p), tile_hi(2 * p + 1));
        float mx = -INFINITY;
        for (int s = 0; s < a.S; ++s) {
            const int lo = Tf * s / a.S, jhi = Tf * (s + 1) / a.S;
            if (min(hi_m, jhi) - lo <= 0) continue;
            mx = fmaxf(mx, a.lse_part[((static_cast<size_t>(s) * a.B + b) * a.H + h) * a.N + n]);
        }
        float acc[E];
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = 0.f;
        float wsum = 0.f;
        if (mx != -INFINITY) {
            for (int s = 0; s < a.S; ++s) {
                const int lo = Tf * s / a.S, jhi = Tf * (s + 1) / a.S;
                if (min(hi_m, jhi) - lo <= 0) continue;
                const float ls = a.lse_part[((static_cast<size_t>(s) * a.B + b) * a.H + h) * a.N + n];
                const float w = expf(ls - mx);
                wsum += w;
                const float *src = a.o_part + (((static_cast<size_t>(s) * a.B + b) * a.N + n) * a.H + h) * D
                                   + lane * E;
                if constexpr (E == 2) {
                    const float2 v = *reinterpret_cast<const float2 *>(src);
                    acc[0] = fmaf(w, v.x, acc[0]);
                    acc[1] = fmaf(w, v.y, acc[1]);
                } else {
#pragma unroll
                    for (int e = 0; e < E; e += 4) {
                        const float4 v = *reinterpret_cast<const float4 *>(src + e);
                        acc[e] = fmaf(w, v.x, acc[e]);
                        acc[e + 1] = fmaf(w, v.y, acc[e + 1]);
                        acc[e + 2] = fmaf(w, v.z, acc[e + 2]);
                        acc[e + 3] = fmaf(w, v.w, acc[e + 3]);
                    }
                }
            }
        }
        const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
        uint16_t *dst = reinterpret_cast<uint16_t *>(a.o) + row * D + lane * E;
        uint32_t pk[E / 2];
#pragma unroll
        for (int e = 0; e < E; e += 2) pk[e / 2] = pack2<kBF16>(acc[e] * inv, acc[e + 1] * inv);
        if constexpr (E == 2) {
            *reinterpret_cast<uint32_t *>(dst) = pk[0];
        } else {
            *reinterpret_cast<uint2 *>(dst) = make_uint2(pk[0], pk[1]);
        }
        if (a.lse != nullptr && lane == 0)
            a.lse[(static_cast<size_t>(b) * a.H + h) * a.N + n] =
                wsum > 0.f ? mx + logf(wsum) : -INFINITY;
    }
}

cudaError_t launch_combine(const CombineArgs &a, int grid, cudaStream_t stream) {
    if (a.d == 64)
        a.bf16 ? fa_combine_kernel<64, true><<<grid, 256, 0, stream>>>(a)
               : fa_combine_kernel<64, false><<<grid, 256, 0, stream>>>(a);
    else
        a.bf16 ? fa_combine_kernel<128, true><<<grid, 256, 0, stream>>>(a)
               : fa_combine_kernel<128, false><<<grid, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace fa
