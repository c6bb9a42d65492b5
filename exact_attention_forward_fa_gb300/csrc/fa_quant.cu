// fa_quant.cu -- FP8 e4m3 block quantization with optional incoherent
// processing, the pre-pass of the FP8 forward.
//
// "FlashAttention-3 on Hopper", sec. 6.3 (block quantization: one FP32
// scale per 128-row tile of a head) and sec. 6.4 (incoherent processing:
// x <- x M with M = (1/sqrt d) H D, H the Sylvester Hadamard matrix, D a
// diagonal of +-1, evaluated as a fast Walsh-Hadamard transform).
//
// Memory-bound (reads 2 B and writes 1 B per element), so both kernels are
// built around keeping HBM busy: persistent CTAs walk the (b, h, 128-row
// tile) list; each tile arrives by TMA into a two-stage shared-memory ring,
// so the next tile is in flight while this one is transformed, reduced and
// stored.  The tile's amax is reduced through shared memory; scale = amax /
// 448 (1 for an all-zero tile); codes = e4m3(y * (1 / scale)), the FP32
// reciprocal formed once per tile (within one rounding of y / scale), round
// to nearest even with saturation.
//   * Without rotation (fa_quantize_kernel): 256 threads, warp w owns rows
//     16w .. 16w+15, lane l holds elements [l*E, l*E + E) of a row (E = d/32),
//     so a warp stores a whole row of codes at once.
//   * With rotation (fa_quantize_rot_kernel): one thread per row (two at
//     d = 256), holding up to 128 elements, so the Walsh-Hadamard butterflies
//     stay in registers; only the top index bit at d = 256 crosses lanes (one
//     shuffle level).  Two threads per row at d = 128 (one shuffle level,
//     twice the warps) measured slower: 24.6 against 22.5 us per tensor.  Spreading a row over a warp instead (as above) took five
//     shuffle levels per element and made the pass issue-bound at 0.42 of
//     HBM.  The tile arrives in TMA's 128-byte swizzle, so the threads' row
//     reads from shared memory do not conflict; the codes are staged the same
//     way and written by TMA stores (a thread storing its own row from
//     registers touched 32 rows per warp instruction).  The butterflies run
//     over the index bits from the lowest up, the same order in either
//     layout.
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
    static constexpr int min_blocks() { return D == 256 ? 1 : 3; }
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

template <int D, int kMode>
__global__ void __launch_bounds__(256, QuantCfg<D>::min_blocks())
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

// ---------------------------------------------------------------------------
// Rotated pre-pass, one thread per row (two at d = 256).
// ---------------------------------------------------------------------------
template <int D>
struct RotCfg {
    static constexpr int E = D > 128 ? 128 : D;        // elements per thread
    static constexpr int TPR = D / E;                  // threads per row: 1, or 2 at d = 256
    static constexpr int NT = 128 * TPR;               // threads per CTA
    static constexpr int NWARP = NT / 32;
    static constexpr int NCH = D / 64;                 // 128-byte chunks of a bf16 row
    static constexpr uint32_t CHUNK = 128u * 128u;     // 128 rows x 128 B
    static constexpr uint32_t TILE_BYTES = NCH * CHUNK;
    static constexpr int NSTAGE = 2;
    // codes of a tile, staged for the TMA store: 128-byte chunks of 128 rows
    // (d >= 128, 128-byte swizzle) or 64-byte rows (d = 64, 64-byte swizzle)
    static constexpr uint32_t CODES_BYTES = 128u * D;
    static constexpr uint32_t CODES_OFF = NSTAGE * TILE_BYTES;
    static constexpr uint32_t SGN_OFF = CODES_OFF + CODES_BYTES;    // float [D]
    static constexpr uint32_t BAR_OFF = SGN_OFF + D * 4;
    static constexpr uint32_t AMAX_OFF = BAR_OFF + 8 * NSTAGE;     // float [2][NWARP]
    static constexpr uint32_t FLAG_OFF = AMAX_OFF + 2 * NWARP * 4;
    static constexpr uint32_t SMEM_BYTES = FLAG_OFF + 16 + 1024;   // + align slack
    static constexpr int BLOCKS = D == 256 ? 1 : D == 128 ? 2 : 4;  // resident CTAs per SM
    // thread -> (row, part): the parts of a row sit in lanes 32 / TPR apart
    // of one warp, so the cross-thread butterflies are warp shuffles
    static constexpr int RPW = 32 / TPR;               // rows per warp
};

template <int D, int kMode>
__global__ void __launch_bounds__(RotCfg<D>::NT, RotCfg<D>::BLOCKS)
fa_quantize_rot_kernel(const __grid_constant__ CUtensorMap tm_x,
                       const __grid_constant__ CUtensorMap tm_x8, const QuantArgs a) {
    using C = RotCfg<D>;
    constexpr int E = C::E;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;   // swizzle atoms
    uint8_t *gbase = smem_raw + (base - smem_addr(smem_raw));
    auto bar = [&](int s) { return base + C::BAR_OFF + 8u * s; };
    float *sgn_s = reinterpret_cast<float *>(gbase + C::SGN_OFF);
    float *warp_amax = reinterpret_cast<float *>(gbase + C::AMAX_OFF);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(gbase + C::FLAG_OFF);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // this thread's row of the tile and part of the row (elements 64 part ..)
    const int row = warp * C::RPW + (lane & (C::RPW - 1));
    const int half = lane / C::RPW;
    const int stride = gridDim.x;

    // thread 0: local step of the last copy issued on each stage (-1: none)
    static_assert(C::NSTAGE == 2, "two stages");
    int last_k0 = -1, last_k1 = -1;
    bool stores_pending = false;           // thread 0: a codes store not yet read
    auto issue = [&](int s, int tile, int kk) {
        if (s == 0) last_k0 = kk; else last_k1 = kk;
        const int tn = tile % a.n_tiles, bh = tile / a.n_tiles;
        mbar_arrive_expect_tx(bar(s), C::TILE_BYTES);
#pragma unroll
        for (int c = 0; c < C::NCH; ++c)
            tma_load_4d(&tm_x, base + s * C::TILE_BYTES + c * C::CHUNK, bar(s), c * 64,
                        bh % a.H, tn * 128, bh / a.H);
    };
    if (tid == 0) {
        *abort_flag = 0u;
        for (int s = 0; s < C::NSTAGE; ++s) mbar_init(bar(s), 1);
        fence_barrier_init();
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_x8);
    }
    // the rotation's diagonal times 1/sqrt(d), correctly rounded to float
    const float inv_sqrt_d = D == 64 ? 0.125f : D == 256 ? 0.0625f : 0.0883883476483184405f;
    for (int i = tid; i < D; i += C::NT) sgn_s[i] = a.signs[i] * inv_sqrt_d;
    __syncthreads();
    if (tid == 0) {
        for (int s = 0; s < C::NSTAGE; ++s) {
            const int tile = blockIdx.x + s * stride;
            if (tile < a.total) issue(s, tile, s);
        }
    }

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

        // ---- this thread's E elements of its row: chunk c holds elements
        //      64c .. 64c+63; 16-byte unit u of row r sits at u ^ (r mod 8) ----
        float2 v2[E / 2];                 // elements 2i, 2i+1 in v2[i]
#pragma unroll
        for (int cc = 0; cc < E / 64; ++cc) {
            const uint32_t rb = base + s * C::TILE_BYTES + (half * (E / 64) + cc) * C::CHUNK + row * 128u;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                uint32_t q0, q1, q2, q3;
                asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(q0), "=r"(q1), "=r"(q2), "=r"(q3)
                             : "r"(rb + ((u ^ (row & 7)) << 4)));
                const uint32_t qq[4] = {q0, q1, q2, q3};
#pragma unroll
                for (int i = 0; i < 4; ++i)       // bf16 -> fp32 is exact
                    v2[(cc * 64 + u * 8) / 2 + i] =
                        make_float2(__uint_as_float(qq[i] << 16), __uint_as_float(qq[i] & 0xffff0000u));
            }
        }
        // Every thread holds its row in registers: refill stage s with the
        // tile NSTAGE steps ahead now, so the copy runs while this tile is
        // transformed (the barrier and the proxy fence order the shared-
        // memory reads before the copy's writes).
        __syncthreads();
        if (tid == 0) {
            const int next = tile + C::NSTAGE * stride;
            if (next < a.total) {
                fence_proxy_async_smem();
                issue(s, next, k + C::NSTAGE);
            }
        }
        // ---- Walsh-Hadamard butterflies over the index bits inside the
        //      thread, lowest first: lower a + b, upper a - b.  Bit 0 pairs
        //      the two halves of a float2; from bit 1 up a butterfly pairs
        //      whole float2s, two butterflies per packed add (the same
        //      roundings as one at a time). ----
#pragma unroll
        for (int i = 0; i < E / 2; ++i) {
            const float a0 = v2[i].x, a1 = v2[i].y;
            v2[i] = make_float2(a0 + a1, a0 - a1);
        }
#pragma unroll
        for (int sb = 1; sb < E / 2; sb <<= 1) {
#pragma unroll
            for (int i = 0; i < E / 2; ++i) {
                if ((i & sb) == 0) {
                    const float2 a0 = v2[i], a1 = v2[i + sb];
                    v2[i] = __fadd2_rn(a0, a1);
                    v2[i + sb] = __fadd2_rn(a0, make_float2(-a1.x, -a1.y));
                }
            }
        }
        if constexpr (C::TPR == 2) {
            // the top index bit (the row's halves, lanes RPW apart): the
            // lower half a + b, the upper a - b, as one fused multiply-add
            // with a +-1 factor (the product is exact)
            const float sl = half ? -1.f : 1.f;
#pragma unroll
            for (int i = 0; i < E / 2; ++i) {
                const float ox = __shfl_xor_sync(0xffffffffu, v2[i].x, C::RPW);
                const float oy = __shfl_xor_sync(0xffffffffu, v2[i].y, C::RPW);
                v2[i] = make_float2(fmaf(v2[i].x, sl, ox), fmaf(v2[i].y, sl, oy));
            }
        }
        // ---- times the signs and 1/sqrt(d); the row's amax ----
        const float4 *sg4 = reinterpret_cast<const float4 *>(sgn_s + half * E);
        float am0 = 0.f, am1 = 0.f;
#pragma unroll
        for (int i = 0; i < E / 4; ++i) {
            const float4 g = sg4[i];
            v2[2 * i] = __fmul2_rn(v2[2 * i], make_float2(g.x, g.y));
            v2[2 * i + 1] = __fmul2_rn(v2[2 * i + 1], make_float2(g.z, g.w));
            am0 = max3(am0, fabsf(v2[2 * i].x), fabsf(v2[2 * i].y));
            am1 = max3(am1, fabsf(v2[2 * i + 1].x), fabsf(v2[2 * i + 1].y));
        }
        float amax = fmaxf(am0, am1);
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
        float *wa = warp_amax + (k & 1) * C::NWARP;
        if (lane == 0) wa[warp] = amax;
        // the codes buffer must have been read by the previous tile's store
        if (kMode != kScalesOnly && tid == 0 && stores_pending) {
            bulk_wait_read();
            stores_pending = false;
        }
        __syncthreads();
        float tmax = wa[0];
#pragma unroll
        for (int i = 1; i < C::NWARP; ++i) tmax = fmaxf(tmax, wa[i]);
        float scale = tmax > 0.f ? tmax / 448.f : 1.f;
        if constexpr (kMode == kGiven) scale = a.scale_in[static_cast<size_t>(bh) * a.n_tiles + tn];
        const float inv = 1.f / scale;
        if (kMode != kGiven && tid == 0) a.scales[static_cast<size_t>(bh) * a.n_tiles + tn] = scale;
        if constexpr (kMode == kScalesOnly) continue;

        // ---- codes into the staging buffer (row r's 16-byte unit u at
        //      u ^ (r mod 8) in 128-byte lines, u ^ ((r / 2) mod 4) in the
        //      64-byte rows of d = 64: the swizzles the TMA store undoes) ----
        const float2 inv2 = make_float2(inv, inv);
#pragma unroll
        for (int g = 0; g < E / 16; ++g) {
            uint32_t w4[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint16_t lo, hi;
                const int e2 = (g * 16 + 4 * i) / 2;
                const float2 y01 = __fmul2_rn(v2[e2], inv2);
                const float2 y23 = __fmul2_rn(v2[e2 + 1], inv2);
                asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(y01.y), "f"(y01.x));
                asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(y23.y), "f"(y23.x));
                w4[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
            }
            uint32_t dst;
            if constexpr (D == 64) {
                dst = base + C::CODES_OFF + row * 64u + ((g ^ ((row >> 1) & 3)) << 4);
            } else {
                // 128 codes per 128-byte line, chunk `half` at d = 256
                dst = base + C::CODES_OFF + half * C::CHUNK + row * 128u + ((g ^ (row & 7)) << 4);
            }
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};"
                         :: "r"(dst), "r"(w4[0]), "r"(w4[1]), "r"(w4[2]), "r"(w4[3]) : "memory");
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            // rows >= N fall outside the tensor and are not written
#pragma unroll
            for (int c8 = 0; c8 < (D == 64 ? 1 : D / 128); ++c8)
                tma_store_4d(&tm_x8, base + C::CODES_OFF + c8 * C::CHUNK, c8 * 128, h, tn * 128, b);
            bulk_commit();
            stores_pending = true;
        }
    }
    // Let every copy thread 0 issued land, and its stores complete, before
    // the CTA can exit.
    if (tid == 0) {
        if (last_k0 >= 0) mbar_wait_quiet(bar(0), static_cast<uint32_t>(last_k0 / 2) & 1u, 500000000ull);
        if (last_k1 >= 0) mbar_wait_quiet(bar(1), static_cast<uint32_t>(last_k1 / 2) & 1u, 500000000ull);
        bulk_wait_all();
    }
}

template <int D, int kMode>
static cudaError_t launch_quantize_rot_d(const QuantLaunch &L) {
    using C = RotCfg<D>;
    auto kern = fa_quantize_rot_kernel<D, kMode>;
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
    const int grid = min(L.args.total, L.sm_count * C::BLOCKS);
    kern<<<grid, C::NT, C::SMEM_BYTES, L.stream>>>(L.x, L.x8, L.args);
    return cudaGetLastError();
}

template <int D, int kMode>
static cudaError_t launch_quantize_d(const QuantLaunch &L) {
    using C = QuantCfg<D>;
    auto kern = fa_quantize_kernel<D, kMode>;
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
    const int grid = min(L.args.total, L.sm_count * C::min_blocks());
    kern<<<grid, 256, C::SMEM_BYTES, L.stream>>>(L.x, L.args);
    return cudaGetLastError();
}

// The rotated pass takes the map with 64-element boxes and the 128-byte
// swizzle, the plain pass the map with whole-row boxes (QuantLaunch.x).
template <int kMode>
static cudaError_t launch_quantize_pass(const QuantLaunch &L) {
    const bool rot = L.args.signs != nullptr;
    if (L.d == 64)
        return rot ? launch_quantize_rot_d<64, kMode>(L) : launch_quantize_d<64, kMode>(L);
    if (L.d == 128)
        return rot ? launch_quantize_rot_d<128, kMode>(L) : launch_quantize_d<128, kMode>(L);
    return rot ? launch_quantize_rot_d<256, kMode>(L) : launch_quantize_d<256, kMode>(L);
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
