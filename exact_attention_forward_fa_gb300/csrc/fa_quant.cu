// fa_quant.cu -- FP8 e4m3 block quantization with optional incoherent
// processing, the pre-pass of the FP8 forward.
//
// "FlashAttention-3 on Hopper", sec. 6.3 (block quantization: one FP32
// scale per 128-row tile of a head) and sec. 6.4 (incoherent processing:
// x <- x M with M = (1/sqrt d) H D, H the Sylvester Hadamard matrix, D a
// diagonal of +-1, evaluated as a fast Walsh-Hadamard transform).
//
// Memory-bound (reads 2 B and writes 1 B per element), so the kernel is
// built around keeping HBM busy: persistent CTAs walk the (b, h, 128-row
// tile) list; each tile arrives by one TMA copy into a two-stage shared
// memory ring, so the next tile is in flight while this one is transformed,
// reduced and stored.  256 threads: warp w owns rows 16w .. 16w+15 of the
// tile; lane l holds elements [l*E, l*E + E) of a row (E = d/32).  The
// transform runs in registers (butterflies on the index bits inside a lane,
// then across lanes with shuffles).  The tile's amax is reduced through
// shared memory; scale = amax / 448 (1 for an all-zero tile); codes =
// e4m3(y * (1 / scale)), the FP32 reciprocal formed once per tile (within
// one rounding of y / scale), round to nearest even with saturation.
//
// Coarser scales (one per head: the per-(batch, head) descale that the FP8
// forward takes for V; one per tensor: the control of the FA3 numerical-error
// ablation, "without block quantization").  Three launches: the per-tile
// pass above writing only the scales (kScalesOnly), a reduction of those
// scales to their maximum over each head (or the whole tensor), written back
// to every tile of the group, and the pass again with those scales given
// (kGiven), which writes the codes.  The maximum of the per-tile scales is
// the group's amax / 448 exactly: x -> fl(x / 448) is monotonic.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fa_launch.cuh"

namespace fa {

template <int D>
struct QuantCfg {
    static constexpr int E = D / 32;                       // elements per lane per row
    static constexpr int ROWS = 16;                        // rows per warp
    static constexpr uint32_t TILE_BYTES = 128u * D * 2u;  // one bf16 tile
    static constexpr int NSTAGE = 2;
    static constexpr uint32_t BAR_OFF = NSTAGE * TILE_BYTES;
    static constexpr uint32_t AMAX_OFF = BAR_OFF + 8 * NSTAGE;     // float [2][8]
    static constexpr uint32_t FLAG_OFF = AMAX_OFF + 2 * 8 * 4;
    static constexpr uint32_t SMEM_BYTES = FLAG_OFF + 16 + 128;    // + align slack
    // resident CTAs per SM: as many as registers allow without spills
    static constexpr int min_blocks(bool rot) { return D == 256 ? 1 : (rot && D == 128) ? 2 : 3; }
};

// Per-lane slice of one row: E bf16 values in one shared-memory load.
template <int E> struct RawWord;
template <> struct RawWord<2> { using type = uint32_t; };
template <> struct RawWord<4> { using type = uint2; };
template <> struct RawWord<8> { using type = uint4; };

// bf16 -> fp32 is exact: the 16 bits become the high half of the float.
template <int E>
__device__ __forceinline__ void unpack_bf16(const typename RawWord<E>::type &w, float (&v)[E]) {
    uint32_t ws[E / 2];
    if constexpr (E == 2) {
        ws[0] = w;
    } else if constexpr (E == 4) {
        ws[0] = w.x; ws[1] = w.y;
    } else {
        ws[0] = w.x; ws[1] = w.y; ws[2] = w.z; ws[3] = w.w;
    }
#pragma unroll
    for (int i = 0; i < E / 2; ++i) {
        v[2 * i] = __uint_as_float(ws[i] << 16);
        v[2 * i + 1] = __uint_as_float(ws[i] & 0xffff0000u);
    }
}

// kMode: 0 per-tile scales and codes, kGiven (1) codes from given scales,
// kScalesOnly (2) per-tile scales without codes.
constexpr int kGiven = 1, kScalesOnly = 2;

template <int D, bool kRot, int kMode>
__global__ void __launch_bounds__(256, QuantCfg<D>::min_blocks(kRot))
fa_quantize_kernel(const __grid_constant__ CUtensorMap tm_x, const QuantArgs a) {
    using C = QuantCfg<D>;
    constexpr int E = C::E, ROWS = C::ROWS;
    using Raw = typename RawWord<E>::type;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_addr(smem_raw) + 127u) & ~127u;
    uint8_t *gbase = smem_raw + (base - smem_addr(smem_raw));
    auto bar = [&](int s) { return base + C::BAR_OFF + 8u * s; };
    float *warp_amax = reinterpret_cast<float *>(gbase + C::AMAX_OFF);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(gbase + C::FLAG_OFF);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int stride = gridDim.x;

    // thread 0: local step of the last copy issued on each stage (-1: none)
    static_assert(C::NSTAGE == 2, "two stages");
    int last_k0 = -1, last_k1 = -1;
    auto issue = [&](int s, int tile, int kk) {
        if (s == 0) last_k0 = kk; else last_k1 = kk;
        const int tn = tile % a.n_tiles, bh = tile / a.n_tiles;
        mbar_arrive_expect_tx(bar(s), C::TILE_BYTES);
        tma_load_4d(&tm_x, base + s * C::TILE_BYTES, bar(s), 0, bh % a.H, tn * 128, bh / a.H);
    };
    if (tid == 0) {
        *abort_flag = 0u;
        for (int s = 0; s < C::NSTAGE; ++s) mbar_init(bar(s), 1);
        fence_barrier_init();
        tma_prefetch_desc(&tm_x);
    }
    __syncthreads();
    if (tid == 0) {
        for (int s = 0; s < C::NSTAGE; ++s) {
            const int tile = blockIdx.x + s * stride;
            if (tile < a.total) issue(s, tile, s);
        }
    }

    // 1/sqrt(d), correctly rounded to float
    const float inv_sqrt_d = D == 64 ? 0.125f : D == 256 ? 0.0625f : 0.0883883476483184405f;
    float sgn[E];
#pragma unroll
    for (int e = 0; e < E; ++e) sgn[e] = kRot ? a.signs[lane * E + e] * inv_sqrt_d : 1.f;

    WaitCtx w{abort_flag, a.status, kRoleQuant};
    int k = 0;
    for (int tile = blockIdx.x; tile < a.total; tile += stride, ++k) {
        const int s = k % C::NSTAGE;
        const uint32_t par = static_cast<uint32_t>(k / C::NSTAGE) & 1u;
        // every thread reaches the vote, so a failed wait ends the loop for all
        const bool ok = mbar_wait(bar(s), par, w, 40);
        if (!__syncthreads_and(ok)) break;
        const int tn = tile % a.n_tiles, bh = tile / a.n_tiles;
        const int b = bh / a.H, h = bh % a.H;

        const Raw *rows = reinterpret_cast<const Raw *>(gbase + s * C::TILE_BYTES);
        float y[ROWS][E];
        float amax = 0.f;
#pragma unroll
        for (int rr = 0; rr < ROWS; ++rr) {
            float v[E];
            unpack_bf16<E>(rows[(warp * ROWS + rr) * 32 + lane], v);
            if constexpr (kRot) {
                // Walsh-Hadamard butterflies: index i = lane*E + e.  Bits
                // below log2(E) are inside a lane, the rest select the lane.
#pragma unroll
                for (int sb = 1; sb < E; sb <<= 1) {
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        if ((e & sb) == 0) {
                            const float a0 = v[e], a1 = v[e + sb];
                            v[e] = a0 + a1;
                            v[e + sb] = a0 - a1;
                        }
                    }
                }
                // across lanes: lower lane a + b, upper lane a - b, as one
                // fused multiply-add with a +-1 factor (the product is exact)
#pragma unroll
                for (int m = 1; m < 32; m <<= 1) {
                    const float sl = (lane & m) ? -1.f : 1.f;
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        const float other = __shfl_xor_sync(0xffffffffu, v[e], m);
                        v[e] = fmaf(v[e], sl, other);
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
        float *wa = warp_amax + (k & 1) * 8;
        if (lane == 0) wa[warp] = amax;
        __syncthreads();
        // Stage s has been read by every thread: refill it with the tile
        // NSTAGE steps ahead (the barrier and the proxy fence order the
        // shared-memory reads before the copy's writes).
        if (tid == 0) {
            const int next = tile + C::NSTAGE * stride;
            if (next < a.total) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issue(s, next, k + C::NSTAGE);
            }
        }
        float tmax = wa[0];
#pragma unroll
        for (int i = 1; i < 8; ++i) tmax = fmaxf(tmax, wa[i]);
        float scale = tmax > 0.f ? tmax / 448.f : 1.f;
        if constexpr (kMode == kGiven) scale = a.scale_in[static_cast<size_t>(bh) * a.n_tiles + tn];
        const float inv = 1.f / scale;
        if (kMode != kGiven && tid == 0) a.scales[static_cast<size_t>(bh) * a.n_tiles + tn] = scale;
        if constexpr (kMode == kScalesOnly) continue;

#pragma unroll
        for (int rr = 0; rr < ROWS; ++rr) {
            const int n = tn * 128 + warp * ROWS + rr;
            if (n >= a.N) continue;
            uint8_t *dst = a.x8 + ((static_cast<size_t>(b) * a.N + n) * a.H + h) * D + lane * E;
            uint32_t packed[E / 2];
#pragma unroll
            for (int e = 0; e < E; e += 2) {
                uint16_t pr;
                asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pr)
                    : "f"(y[rr][e + 1] * inv), "f"(y[rr][e] * inv));
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
    // Let every copy thread 0 issued land before the CTA can exit (local
    // step k used stage k % NSTAGE and phase k / NSTAGE of its barrier).
    if (tid == 0) {
        if (last_k0 >= 0) mbar_wait_quiet(bar(0), static_cast<uint32_t>(last_k0 / 2) & 1u, 500000000ull);
        if (last_k1 >= 0) mbar_wait_quiet(bar(1), static_cast<uint32_t>(last_k1 / 2) & 1u, 500000000ull);
    }
}

template <int D, bool kRot, int kMode>
static cudaError_t launch_quantize_d(const QuantLaunch &L) {
    using C = QuantCfg<D>;
    auto kern = fa_quantize_kernel<D, kRot, kMode>;
    static unsigned long long configured = 0ull;   // bit per device id (< 64)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(__atomic_load_n(&configured, __ATOMIC_ACQUIRE) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(C::SMEM_BYTES));
        if (e != cudaSuccess) return e;
        __atomic_fetch_or(&configured, bit, __ATOMIC_ACQ_REL);
    }
    const int grid = min(L.args.total, L.sm_count * C::min_blocks(kRot));
    kern<<<grid, 256, C::SMEM_BYTES, L.stream>>>(L.x, L.args);
    return cudaGetLastError();
}

template <int kMode>
static cudaError_t launch_quantize_pass(const QuantLaunch &L) {
    const bool rot = L.args.signs != nullptr;
    if (L.d == 64)
        return rot ? launch_quantize_d<64, true, kMode>(L) : launch_quantize_d<64, false, kMode>(L);
    if (L.d == 128)
        return rot ? launch_quantize_d<128, true, kMode>(L) : launch_quantize_d<128, false, kMode>(L);
    return rot ? launch_quantize_d<256, true, kMode>(L) : launch_quantize_d<256, false, kMode>(L);
}

// One CTA per group of n consecutive scales: all of them become the
// group's maximum.
__global__ void __launch_bounds__(256)
fa_scale_group_max_kernel(float *scales, long long n) {
    __shared__ float part[8];
    float *g = scales + static_cast<long long>(blockIdx.x) * n;
    float m = 0.f;
    for (long long i = threadIdx.x; i < n; i += 256) m = fmaxf(m, g[i]);
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, k));
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = m;
    __syncthreads();
    m = part[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) m = fmaxf(m, part[i]);
    for (long long i = threadIdx.x; i < n; i += 256) g[i] = m;
}

cudaError_t launch_quantize(const QuantLaunch &L) {
    if (L.granularity == 0) return launch_quantize_pass<0>(L);
    cudaError_t e = launch_quantize_pass<kScalesOnly>(L);
    if (e != cudaSuccess) return e;
    // one group per head, or one for the whole tensor
    const long long groups = L.granularity == 1 ? static_cast<long long>(L.args.B) * L.args.H : 1;
    const long long n = static_cast<long long>(L.args.total) / groups;
    fa_scale_group_max_kernel<<<static_cast<unsigned>(groups), 256, 0, L.stream>>>(L.args.scales, n);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    QuantLaunch G = L;
    G.args.scale_in = L.args.scales;
    return launch_quantize_pass<kGiven>(G);
}

}  // namespace fa
