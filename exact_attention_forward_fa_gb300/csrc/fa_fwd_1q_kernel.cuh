// fa_fwd_1q_kernel.cuh -- exact attention forward, one Q tile per work unit
// (used for head dim 256) on sm_103a.
//
// Same operation as fa_fwd_kernel.cuh ("FlashAttention-3 on Hopper",
// sec. 4.1-4.7: online softmax over key tiles, LSE in natural-log units,
// bottom-right causal predicate), scheduled for d = 256 where the output
// accumulator alone is 256 TMEM columns per 128-row Q tile:
//   * one 128-row Q tile per work unit, BN-key K/V tiles (BN = 64 at d = 256,
//     128 otherwise; measured slower than the two-tile kernel at d <= 128,
//     where one softmax warpgroup cannot keep up with the tensor core);
//   * TMEM (512 columns): S0 [0,BN), S1 [BN,2BN) double-buffered scores (P
//     overlays the first BN/2 columns of its S buffer), Q [2BN, 2BN+d/2) as
//     the A operand of S = Q K^T (TS form, so Q is not re-read from shared
//     memory for every key tile), O after it (at d = 256: [256,512));
//   * shared memory: a 64 KB Q staging tile (TMA, 128-byte swizzle) that the
//     softmax threads copy into TMEM, and a 5-stage ring of 32 KB K/V tiles;
//   * MMA order QK(t), PV(t-1): the score tile of step t+1 is computed while
//     the softmax of step t runs ("FlashAttention v1-v4", FA4 forward
//     schedule: S in TMEM, softmax, P back to TMEM, PV);
//   * conditional rescale with tau = 8 ("FlashAttention v1-v4", conditional
//     rescale); the O correction waits for the previous PV to complete.
// Warps: 0-3 softmax (thread = row = TMEM lane; also the Q copy and the
// epilogue), 4 TMA producer (one lane), 5 MMA issuer (converged warp,
// elect.sync issue).  Every mbarrier wait is bounded.
#pragma once

#include "fa_device.cuh"
#include "fa_fwd_kernel.cuh"   // FwdArgs

namespace fa {

template <int D, bool kCausal, bool kBF16>
struct Fwd1qCfg {
    static_assert(D == 64 || D == 128 || D == 256, "head dim");
    static constexpr int BM = 128;
    static constexpr int BN = (D == 256) ? 64 : 128;           // keys per tile
    static constexpr int NCH = D / 64;                          // 128-B column chunks
    static constexpr uint32_t Q_CHUNK = 128u * 128u;            // 128 rows x 128 B
    static constexpr uint32_t KV_CHUNK = BN * 128u;             // BN rows x 128 B
    static constexpr uint32_t Q_BYTES = NCH * Q_CHUNK;
    static constexpr uint32_t KV_BYTES = NCH * KV_CHUNK;
    static constexpr int NSTAGE = (D == 256) ? 5 : (D == 128) ? 6 : 8;
    static constexpr int NTHREADS = 192;

    static constexpr uint32_t QS_OFF = 0;
    static constexpr uint32_t KV_OFF = Q_BYTES;
    static constexpr uint32_t BAR_OFF = KV_OFF + NSTAGE * KV_BYTES;
    static constexpr int B_QSFULL = 0, B_QSEMPTY = 1, B_QTFULL = 2, B_KVFULL = 3,
                         B_KVEMPTY = B_KVFULL + NSTAGE, B_SFULL = B_KVEMPTY + NSTAGE,
                         B_PFULL = B_SFULL + 2, B_PVDONE = B_PFULL + 2,
                         B_OEMPTY = B_PVDONE + 1, B_MMADONE = B_OEMPTY + 1,
                         // causal: the dynamic order's answers (see the kernel)
                         B_CLCFULL = B_MMADONE + 1, B_UNIT = B_CLCFULL + 4,
                         B_CLCEMPTY = B_UNIT + 4, NBAR = B_CLCEMPTY + 4;
    static constexpr int CLC_DEPTH = 4;
    static constexpr uint32_t MISC_OFF = BAR_OFF + NBAR * 8;
    static constexpr uint32_t CLC_OFF = (MISC_OFF + 16 + 15) & ~15u;   // 16-byte aligned
    static constexpr uint32_t UNIT_OFF = CLC_OFF + CLC_DEPTH * 16;
    static constexpr uint32_t SMEM_BYTES = UNIT_OFF + CLC_DEPTH * 4 + 1024;
    static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");

    // TMEM: S0 [0,BN), S1 [BN,2BN), Q [2BN, 2BN + D/2), O [.., + D)
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_Q = 2 * BN, COL_O = 2 * BN + D / 2;
    static_assert(COL_O + D <= TMEM_COLS, "TMEM budget");
    __host__ __device__ static constexpr uint32_t col_s(int b) { return b ? BN : 0u; }

    static constexpr uint32_t IDESC_QK = idesc_f16(128, BN, kBF16, false, false);
    static constexpr uint32_t IDESC_PV = idesc_f16(128, D, kBF16, false, true);
    static constexpr float TAU = 8.0f;
};

// Work unit: one 128-row Q tile of one (b, h); keys in BN-wide tiles visited
// in descending order from T-1 to 0.
struct Unit1q {
    int b, h, m, T;
};

template <bool kCausal, int BN>
__device__ __forceinline__ Unit1q make_unit_1q(int u, const FwdArgs &a) {
    Unit1q U;
    const int BH = a.B * a.H;
    const int n_qt = (a.N + 127) / 128;
    int bh;
    if (kCausal) {            // the dynamic order of fa_fwd_kernel.cuh
        dynamic_order(u, BH, n_qt, a.chunk, U.m, bh);
    } else {
        U.m = u % n_qt;
        bh = u / n_qt;
    }
    U.b = bh / a.H;
    U.h = bh % a.H;
    // a.n_kv counts BN-key tiles; the diagonal tile holds key m*128 + 127
    U.T = kCausal ? min(a.n_kv, (U.m * 128 + 127) / BN + 1) : a.n_kv;
    return U;
}

template <int D, bool kCausal, bool kBF16>
__global__ void __launch_bounds__(192, 1)
fa_fwd_1q_kernel(const __grid_constant__ CUtensorMap tm_q,
                 const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const FwdArgs a) {
    using C = Fwd1qCfg<D, kCausal, kBF16>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    auto bar = [&](int i) -> uint32_t { return base + C::BAR_OFF + 8u * i; };
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(gbase + C::MISC_OFF);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(gbase + C::MISC_OFF + 4);
    // Causal: the dynamic order of fa_fwd_kernel.cuh (one CTA per unit).  The
    // producer asks for the next unit once it has issued the loads of the
    // current one; the k-th answer goes to slot k % CLC_DEPTH, the producer
    // publishes its block index there (-1: none left), and the MMA warp and
    // the 4 softmax warps read it and release the slot.
    volatile int *unit_slot = reinterpret_cast<volatile int *>(gbase + C::UNIT_OFF);
    if (warp == 5) tmem_alloc(base + C::MISC_OFF, C::TMEM_COLS);
    if (tid == 0) {
        *abort_flag = 0u;
        mbar_init(bar(C::B_QSFULL), 1);
        mbar_init(bar(C::B_QSEMPTY), 4);
        mbar_init(bar(C::B_QTFULL), 4);
        for (int s = 0; s < C::NSTAGE; ++s) {
            mbar_init(bar(C::B_KVFULL + s), 1);
            mbar_init(bar(C::B_KVEMPTY + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(C::B_SFULL + b), 1);
            mbar_init(bar(C::B_PFULL + b), 4);
        }
        mbar_init(bar(C::B_PVDONE), 1);
        mbar_init(bar(C::B_OEMPTY), 4);
        mbar_init(bar(C::B_MMADONE), 1);
        for (int q = 0; kCausal && q < C::CLC_DEPTH; ++q) {
            mbar_init(bar(C::B_CLCFULL + q), 1);
            mbar_init(bar(C::B_UNIT + q), 1);
            mbar_init(bar(C::B_CLCEMPTY + q), 5);
        }
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;

    if (warp == 4) {
        // =================== TMA producer (one lane) ===================
        if (lane == 0) {
            WaitCtx w{abort_flag, a.status, kRoleProducer};
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            uint32_t slot = 0, phase = 0, armed = 0, armed_par = 0;
            int qn = 0;
            bool ok = true;
            auto load_kv = [&](const CUtensorMap *tm, const Unit1q &U, int j) -> bool {
                if (!mbar_wait(bar(C::B_KVEMPTY + slot), phase ^ 1, w, 2)) return false;
                mbar_arrive_expect_tx(bar(C::B_KVFULL + slot), C::KV_BYTES);
#pragma unroll
                for (int c = 0; c < C::NCH; ++c)
                    tma_load_4d(tm, base + C::KV_OFF + slot * C::KV_BYTES + c * C::KV_CHUNK,
                                bar(C::B_KVFULL + slot), c * 64, U.h / a.group, j * C::BN, U.b);
                armed |= 1u << slot;
                armed_par = (armed_par & ~(1u << slot)) | (phase << slot);
                if (++slot == C::NSTAGE) { slot = 0; phase ^= 1; }
                return true;
            };
            uint32_t kq = 0;                        // causal: requests issued
            bool clc_pending = false;
            auto next_u = [&]() __attribute__((always_inline)) -> int {
                    if (!ok) return -1;
                const uint32_t q = kq % C::CLC_DEPTH, ph = (kq / C::CLC_DEPTH) & 1u;
                ++kq;
                if (!mbar_wait(bar(C::B_CLCEMPTY + q), ph ^ 1u, w, 3)) { ok = false; return -1; }
                mbar_arrive_expect_tx(bar(C::B_CLCFULL + q), 16u);
                clc_try_cancel(base + C::CLC_OFF + 16u * q, bar(C::B_CLCFULL + q));
                clc_pending = true;
                if (!mbar_wait(bar(C::B_CLCFULL + q), ph, w, 4)) { ok = false; return -1; }
                clc_pending = false;
                const int nu = clc_block(base + C::CLC_OFF + 16u * q);
                unit_slot[q] = nu;
                mbar_arrive(bar(C::B_UNIT + q));        // release: the index is visible
                return nu;
            };
            for (int u = blockIdx.x, st = unit_stride0(kCausal); ok && (!kCausal || u >= 0) && u < a.n_units;
                 u = kCausal ? next_u() : u + st, st = 2 * static_cast<int>(gridDim.x) - st) {
                const Unit1q U = make_unit_1q<kCausal, C::BN>(u, a);
                ok = mbar_wait(bar(C::B_QSEMPTY), (qn & 1) ^ 1, w, 1);
                if (!ok) break;
                mbar_arrive_expect_tx(bar(C::B_QSFULL), C::Q_BYTES);
#pragma unroll
                for (int c = 0; c < C::NCH; ++c)
                    tma_load_4d(&tm_q, base + C::QS_OFF + c * C::Q_CHUNK, bar(C::B_QSFULL),
                                c * 64, U.h, U.m * 128, U.b);
                ++qn;
                // ring order = MMA consumption order: K(0), then K(t), V(t-1)
                // for t = 1..T-1, then V(T-1); tile t is key tile j = T-1-t.
                ok = load_kv(&tm_k, U, U.T - 1);
                for (int t = 1; ok && t < U.T; ++t) {
                    ok = load_kv(&tm_k, U, U.T - 1 - t);
                    if (ok) ok = load_kv(&tm_v, U, U.T - t);
                }
                if (ok) ok = load_kv(&tm_v, U, 0);
            }
            if (kCausal && clc_pending)
                mbar_wait_quiet(bar(C::B_CLCFULL + (kq - 1) % C::CLC_DEPTH),
                                ((kq - 1) / C::CLC_DEPTH) & 1u, 500000000ull);
            for (int s = 0; s < C::NSTAGE; ++s)
                if (armed & (1u << s))
                    mbar_wait_quiet(bar(C::B_KVFULL + s), (armed_par >> s) & 1u, 500000000ull);
            if (qn > 0) mbar_wait_quiet(bar(C::B_QSFULL), (qn - 1) & 1, 500000000ull);
        }
        __syncwarp();
    } else if (warp == 5) {
        // =================== MMA issuer (whole warp, elected lane issues) ===================
        WaitCtx w{abort_flag, a.status, kRoleMma};
        uint32_t slot = 0, phase = 0;
        uint32_t pph0 = 0, pph1 = 0, qtph = 0, un = 0;
        bool ok = true;
        auto next_slot = [&](uint32_t &s_out, uint32_t &p_out) {
            s_out = slot;
            p_out = phase;
            if (++slot == C::NSTAGE) { slot = 0; phase ^= 1; }
        };
        uint32_t kq = 0;                            // causal: answers read
        auto next_u = [&]() __attribute__((always_inline)) -> int {
            if (!ok) return -1;
            const uint32_t q = kq % C::CLC_DEPTH, ph = (kq / C::CLC_DEPTH) & 1u;
            ++kq;
            if (!mbar_wait_warp(bar(C::B_UNIT + q), ph, w, 35)) { ok = false; return -1; }
            const int nu = unit_slot[q];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_CLCEMPTY + q));
            return nu;
        };
        for (int u = blockIdx.x, st = unit_stride0(kCausal); ok && (!kCausal || u >= 0) && u < a.n_units;
                 u = kCausal ? next_u() : u + st, st = 2 * static_cast<int>(gridDim.x) - st) {
            const Unit1q U = make_unit_1q<kCausal, C::BN>(u, a);
            ok = mbar_wait_warp(bar(C::B_QTFULL), qtph, w, 30);
            if (!ok) break;
            qtph ^= 1;
            for (int t = 0; t <= U.T && ok; ++t) {
                if (t < U.T) {
                    // ---- S[t%2] = Q K_t^T (A = Q from TMEM) ----
                    uint32_t ks, kp;
                    next_slot(ks, kp);
                    ok = mbar_wait_warp(bar(C::B_KVFULL + ks), kp, w, 31);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t kd = smem_desc_sw128(base + C::KV_OFF + ks * C::KV_BYTES, 16u, 1024u);
                    const uint32_t sb = t & 1;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = ((kk >> 2) * C::KV_CHUNK + (kk & 3) * 32u) >> 4;
                        mma_ts_f16_elect(tbase + C::col_s(sb), tbase + C::COL_Q + kk * 8u, kd + off,
                                         C::IDESC_QK, kk > 0 ? 1u : 0u);
                    }
                    mma_commit_elect(bar(C::B_SFULL + sb));
                    mma_commit_elect(bar(C::B_KVEMPTY + ks));
                }
                if (t >= 1) {
                    // ---- O += P[(t-1)%2] V_(t-1) ----
                    uint32_t vs, vp;
                    next_slot(vs, vp);
                    const uint32_t pb = (t - 1) & 1;
                    ok = mbar_wait_warp(bar(C::B_KVFULL + vs), vp, w, 32);
                    if (ok && t == 1) ok = mbar_wait_warp(bar(C::B_OEMPTY), (un & 1) ^ 1, w, 33);
                    if (ok) ok = mbar_wait_warp(bar(C::B_PFULL + pb), pb ? pph1 : pph0, w, 34);
                    if (!ok) break;
                    if (pb) pph1 ^= 1; else pph0 ^= 1;
                    tc_fence_after();
                    const uint64_t vd = smem_desc_sw128(base + C::KV_OFF + vs * C::KV_BYTES, C::KV_CHUNK, 1024u);
#pragma unroll
                    for (int kk = 0; kk < C::BN / 16; ++kk)
                        mma_ts_f16_elect(tbase + C::COL_O, tbase + C::col_s(pb) + kk * 8u,
                                         vd + ((kk * 2048u) >> 4), C::IDESC_PV,
                                         (t > 1 || kk > 0) ? 1u : 0u);
                    mma_commit_elect(bar(C::B_PVDONE));
                    mma_commit_elect(bar(C::B_KVEMPTY + vs));
                }
            }
            ++un;
        }
        mma_commit_elect(bar(C::B_MMADONE));
        mbar_wait_quiet(bar(C::B_MMADONE), 0, 500000000ull);
        __syncwarp();
    } else {
        // =================== softmax group (warps 0-3) ===================
        const int row = tid;                                     // TMEM lane == tile row
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        const uint32_t tO = tbase + lane_off + C::COL_O;
        const uint32_t tQ = tbase + lane_off + C::COL_Q;
        WaitCtx w{abort_flag, a.status, kRoleSoftmax0};
        const float sl2 = a.scale_log2;
        const float2 c2 = make_float2(sl2, sl2);
        uint32_t sph0 = 0, sph1 = 0, pvph = 0, qsph = 0;
        bool ok = true;
        bool pending_epi = false;
        Unit1q P{};                      // the unit whose epilogue is pending
        float P_le = 0.f, P_lr = 0.f, P_r = -INFINITY;

        auto epilogue = [&]() -> bool {
            // O of unit P is final once its last PV completed.
            if (!mbar_wait(bar(C::B_PVDONE), pvph, w, 41)) return false;
            pvph ^= 1;
            if (__any_sync(0xffffffffu, *abort_flag != 0u)) return false;
            tc_fence_after();
            const bool live = (P_le > 0.f) && (P_lr > 0.f);
            const float inv = live ? 1.f / P_lr : 0.f;
            const int grow = P.m * 128 + row;
            uint16_t *orow = reinterpret_cast<uint16_t *>(a.o) +
                             ((static_cast<size_t>(P.b) * a.N + grow) * a.H + P.h) * D;
#pragma unroll 1
            for (int ch = 0; ch < D / 32; ++ch) {
                uint32_t ov[32];
                tmem_ld32(tO + ch * 32, ov);
                tmem_ld_wait();
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    pk[i] = pack2<kBF16>(__uint_as_float(ov[2 * i]) * inv,
                                         __uint_as_float(ov[2 * i + 1]) * inv);
                if (grow < a.N) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + ch * 32);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_OEMPTY));
            if (a.lse != nullptr && grow < a.N) {
                const float lse = live ? (P_r + log2f(P_le)) * 0.69314718055994530942f : -INFINITY;
                a.lse[(static_cast<size_t>(P.b) * a.H + P.h) * a.N + grow] = lse;
            }
            return true;
        };
        uint32_t kq = 0;                            // causal: answers read
        // (a failed wait leaves this loop by break, so ok holds here)
        auto next_u = [&]() __attribute__((always_inline)) -> int {
            const uint32_t q = kq % C::CLC_DEPTH, ph = (kq / C::CLC_DEPTH) & 1u;
            ++kq;
            ok = mbar_wait(bar(C::B_UNIT + q), ph, w, 45);
            if (__any_sync(0xffffffffu, !ok)) { ok = false; return -1; }
            const int nu = unit_slot[q];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_CLCEMPTY + q));
            return nu;
        };
        for (int u = blockIdx.x, st = unit_stride0(kCausal); ok && (!kCausal || u >= 0) && u < a.n_units;
                 u = kCausal ? next_u() : u + st, st = 2 * static_cast<int>(gridDim.x) - st) {
            const Unit1q U = make_unit_1q<kCausal, C::BN>(u, a);
            // ---- copy Q (staged by TMA, 128-B swizzle) into TMEM; the last
            //      QK of the previous unit completed before its S_FULL ----
            ok = mbar_wait(bar(C::B_QSFULL), qsph, w, 40);
            if (__any_sync(0xffffffffu, !ok)) { ok = false; break; }
            qsph ^= 1;
#pragma unroll 1
            for (int c = 0; c < C::NCH; ++c) {
                uint32_t qv[32];
                const uint32_t rbase = base + C::QS_OFF + c * C::Q_CHUNK + row * 128u;
#pragma unroll
                for (int uu = 0; uu < 8; ++uu) {
                    const uint32_t addr = rbase + ((uu ^ (row & 7)) << 4);
                    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(qv[4 * uu]), "=r"(qv[4 * uu + 1]), "=r"(qv[4 * uu + 2]),
                                   "=r"(qv[4 * uu + 3])
                                 : "r"(addr));
                }
                tmem_st32(tQ + c * 32, qv);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar(C::B_QSEMPTY));
                mbar_arrive(bar(C::B_QTFULL));
            }
            // ---- epilogue of the previous unit, overlapped with this unit's
            //      first score tiles ----
            if (pending_epi) {
                ok = epilogue();
                if (__any_sync(0xffffffffu, !ok)) { ok = false; break; }
                pending_epi = false;
            }
            float r = -INFINITY, le = 0.f, lr = 0.f;
            for (int t = 0; t < U.T; ++t) {
                const int j = U.T - 1 - t;
                const uint32_t sb = t & 1;
                ok = mbar_wait(bar(C::B_SFULL + sb), sb ? sph1 : sph0, w, 42);
                if (__any_sync(0xffffffffu, !ok)) { ok = false; break; }
                if (sb) sph1 ^= 1; else sph0 ^= 1;
                tc_fence_after();
                const uint32_t tS = tbase + lane_off + C::col_s(sb);
                constexpr int BN = C::BN;
                uint32_t s[BN];
#pragma unroll
                for (int c = 0; c < BN; c += 32)
                    tmem_ld32(tS + c, *reinterpret_cast<uint32_t(*)[32]>(&s[c]));
                tmem_ld_wait();
                float *sf = reinterpret_cast<float *>(s);
                // ---- masks: sequence tail and causal diagonal ----
                int lim = BN;
                if (j == a.n_kv - 1) lim = min(lim, a.N - j * BN);
                if (kCausal) lim = min(lim, U.m * 128 + row - j * BN + 1);
                if (lim < BN) {
#pragma unroll
                    for (int c = 0; c < BN; ++c) if (c >= lim) sf[c] = -INFINITY;
                }
                float m0 = sf[0], m1 = sf[1], m2 = sf[2], m3 = sf[3];
#pragma unroll
                for (int c = 4; c < BN; c += 8) {
                    m0 = max3(m0, sf[c + 0], sf[c + 4]);
                    m1 = max3(m1, sf[c + 1], sf[c + 5]);
                    m2 = max3(m2, sf[c + 2], sf[c + 6]);
                    m3 = max3(m3, sf[c + 3], sf[c + 7]);
                }
                const float mx = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
                const float bnew = mx * sl2;
                float rn, corr;
                if (r == -INFINITY) { rn = bnew; corr = 1.f; }
                else { rn = (bnew > r + C::TAU) ? bnew : r; corr = ex2_approx(r - rn); }
                const bool need = (r != -INFINITY) && (rn != r);
                const float rs = (rn == -INFINITY) ? 0.f : rn;
                const float2 nr2 = make_float2(-rs, -rs);
                float2 e_a = make_float2(0.f, 0.f), e_b = e_a, r_a = e_a, r_b = e_a;
                uint32_t p[BN / 2];
#pragma unroll
                for (int c = 0; c < BN; c += 4) {
                    const float2 x01 = __ffma2_rn(make_float2(sf[c + 0], sf[c + 1]), c2, nr2);
                    const float2 x23 = __ffma2_rn(make_float2(sf[c + 2], sf[c + 3]), c2, nr2);
                    const float2 e01 = make_float2(ex2_approx(x01.x), ex2_approx(x01.y));
                    const float2 e23 = make_float2(ex2_approx(x23.x), ex2_approx(x23.y));
                    const uint32_t pk0 = pack2<kBF16>(e01.x, e01.y);
                    const uint32_t pk1 = pack2<kBF16>(e23.x, e23.y);
                    p[c / 2] = pk0;
                    p[c / 2 + 1] = pk1;
                    e_a = __fadd2_rn(e_a, e01);
                    e_b = __fadd2_rn(e_b, e23);
                    add_pair<kBF16>(r_a.x, r_a.y, pk0);
                    add_pair<kBF16>(r_b.x, r_b.y, pk1);
                }
                le = __fmaf_rn(le, corr, (e_a.x + e_a.y) + (e_b.x + e_b.y));
                lr = __fmaf_rn(lr, corr, (r_a.x + r_a.y) + (r_b.x + r_b.y));
#pragma unroll
                for (int c = 0; c < BN / 2; c += 32)
                    tmem_st32(tS + c, *reinterpret_cast<uint32_t(*)[32]>(&p[c]));
                // ---- the previous PV must be complete before O is rescaled
                //      and before this tile's P is published (one wait per PV) ----
                if (t > 0) {
                    ok = mbar_wait(bar(C::B_PVDONE), pvph, w, 43);
                    if (__any_sync(0xffffffffu, !ok)) { ok = false; break; }
                    pvph ^= 1;
                    tc_fence_after();
                }
                if (__any_sync(0xffffffffu, need)) {
                    const float2 cc = make_float2(corr, corr);
#pragma unroll 1
                    for (int ch = 0; ch < D / 32; ++ch) {
                        uint32_t ov[32];
                        tmem_ld32(tO + ch * 32, ov);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            const float2 v2 = __fmul2_rn(
                                make_float2(__uint_as_float(ov[i]), __uint_as_float(ov[i + 1])), cc);
                            ov[i] = __float_as_uint(v2.x);
                            ov[i + 1] = __float_as_uint(v2.y);
                        }
                        tmem_st32(tO + ch * 32, ov);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::B_PFULL + sb));
                r = rn;
            }
            if (!ok) break;
            P = U;
            P_le = le;
            P_lr = lr;
            P_r = r;
            pending_epi = true;
        }
        if (ok && pending_epi) ok = epilogue();
    }

    // ---- teardown ----
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tbase, C::TMEM_COLS);
    }
}

}  // namespace fa
