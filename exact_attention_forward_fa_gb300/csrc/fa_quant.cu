// fa_quant.cu -- FP8 e4m3 block quantization with optional incoherent
// processing, the pre-pass of the FP8 forward.
//
// "FlashAttention-3 on Hopper", sec. 6.3 (block quantization: one FP32
// scale per 128-row tile of a head) and sec. 6.4 (incoherent processing:
// x <- x M with M = (1/sqrt d) H D, H the Sylvester Hadamard matrix, D a
// diagonal of +-1, evaluated as a fast Walsh-Hadamard transform).
//
// One CTA per (b, h, 128-row tile), 256 threads: warp w owns rows
// 16w .. 16w+15 of the tile; lane l holds elements [l*E, l*E + E) of a row
// (E = d/32).  The transform runs in registers: butterflies on the index
// bits inside a lane, then across lanes with shuffles.  The tile's amax is
// reduced through shared memory; scale = amax / 448 (1 for an all-zero
// tile); codes = e4m3(y / scale), round to nearest even with saturation.
// Memory-bound: reads 2 B and writes 1 B per element.
#include <cuda_runtime.h>

#include <cstdint>

#include "fa_launch.cuh"

namespace fa {

template <int D>
__global__ void __launch_bounds__(256)
fa_quantize_kernel(const uint16_t *__restrict__ x, uint8_t *__restrict__ x8,
                   float *__restrict__ scales, const float *__restrict__ signs,
                   int B, int H, int N, int n_tiles) {
    constexpr int E = D / 32;                  // elements per lane per row
    constexpr int ROWS = 16;                   // rows per warp
    __shared__ float warp_amax[8];
    const int tile = blockIdx.x % n_tiles;
    const int bh = blockIdx.x / n_tiles;
    const int b = bh / H, h = bh % H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // 1/sqrt(d), correctly rounded to float
    const float inv_sqrt_d = D == 64 ? 0.125f : D == 256 ? 0.0625f : 0.0883883476483184405f;

    float sgn[E];
#pragma unroll
    for (int e = 0; e < E; ++e) sgn[e] = signs ? signs[lane * E + e] * inv_sqrt_d : 1.f;

    float y[ROWS][E];
    float amax = 0.f;
#pragma unroll
    for (int rr = 0; rr < ROWS; ++rr) {
        const int n = tile * 128 + warp * ROWS + rr;
        float v[E];
        if (n < N) {
            const uint16_t *src = x + ((static_cast<size_t>(b) * N + n) * H + h) * D + lane * E;
            if constexpr (E == 2) {
                const uint32_t w = *reinterpret_cast<const uint32_t *>(src);
                v[0] = __uint_as_float(w << 16);
                v[1] = __uint_as_float(w & 0xffff0000u);
            } else if constexpr (E == 4) {
                const uint2 w = *reinterpret_cast<const uint2 *>(src);
                v[0] = __uint_as_float(w.x << 16);
                v[1] = __uint_as_float(w.x & 0xffff0000u);
                v[2] = __uint_as_float(w.y << 16);
                v[3] = __uint_as_float(w.y & 0xffff0000u);
            } else {
                const uint4 w = *reinterpret_cast<const uint4 *>(src);
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    v[2 * i] = __uint_as_float(ws[i] << 16);
                    v[2 * i + 1] = __uint_as_float(ws[i] & 0xffff0000u);
                }
            }
        } else {
#pragma unroll
            for (int e = 0; e < E; ++e) v[e] = 0.f;
        }
        if (signs) {
            // Walsh-Hadamard butterflies: index i = lane*E + e.  Bits below
            // log2(E) are inside a lane, the rest select the lane.
#pragma unroll
            for (int s = 1; s < E; s <<= 1) {
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    if ((e & s) == 0) {
                        const float a0 = v[e], a1 = v[e + s];
                        v[e] = a0 + a1;
                        v[e + s] = a0 - a1;
                    }
                }
            }
#pragma unroll
            for (int m = 1; m < 32; m <<= 1) {
                const bool upper = (lane & m) != 0;
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const float other = __shfl_xor_sync(0xffffffffu, v[e], m);
                    v[e] = upper ? (other - v[e]) : (v[e] + other);
                }
            }
#pragma unroll
            for (int e = 0; e < E; ++e) v[e] *= sgn[e];
        }
#pragma unroll
        for (int e = 0; e < E; ++e) {
            y[rr][e] = v[e];
            amax = fmaxf(amax, fabsf(v[e]));
        }
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
    if (lane == 0) warp_amax[warp] = amax;
    __syncthreads();
    float tmax = warp_amax[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) tmax = fmaxf(tmax, warp_amax[i]);
    const float scale = tmax > 0.f ? tmax / 448.f : 1.f;
    if (threadIdx.x == 0) scales[static_cast<size_t>(bh) * n_tiles + tile] = scale;

#pragma unroll
    for (int rr = 0; rr < ROWS; ++rr) {
        const int n = tile * 128 + warp * ROWS + rr;
        if (n >= N) continue;
        uint8_t *dst = x8 + ((static_cast<size_t>(b) * N + n) * H + h) * D + lane * E;
        uint32_t packed[E / 2];
#pragma unroll
        for (int e = 0; e < E; e += 2) {
            uint16_t pr;
            asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pr)
                : "f"(y[rr][e + 1] / scale), "f"(y[rr][e] / scale));
            packed[e / 2] = pr;
        }
        if constexpr (E == 2) {
            *reinterpret_cast<uint16_t *>(dst) = static_cast<uint16_t>(packed[0]);
        } else if constexpr (E == 4) {
            *reinterpret_cast<uint32_t *>(dst) = packed[0] | (packed[1] << 16);
        } else {
            *reinterpret_cast<uint2 *>(dst) =
                make_uint2(packed[0] | (packed[1] << 16), packed[2] | (packed[3] << 16));
        }
    }
}

cudaError_t launch_quantize(const void *x, void *x8, float *scales, const float *signs,
                            int B, int H, int N, int d, cudaStream_t stream) {
    const int n_tiles = (N + 127) / 128;
    const unsigned grid = static_cast<unsigned>(B) * H * n_tiles;
    const auto *xs = static_cast<const uint16_t *>(x);
    auto *q = static_cast<uint8_t *>(x8);
    if (d == 64)
        fa_quantize_kernel<64><<<grid, 256, 0, stream>>>(xs, q, scales, signs, B, H, N, n_tiles);
    else if (d == 128)
        fa_quantize_kernel<128><<<grid, 256, 0, stream>>>(xs, q, scales, signs, B, H, N, n_tiles);
    else
        fa_quantize_kernel<256><<<grid, 256, 0, stream>>>(xs, q, scales, signs, B, H, N, n_tiles);
    return cudaGetLastError();
}

}  // namespace fa
