// fa_fwd_fp8_1q_kernel.cuh -- FP8 (e4m3) attention forward with one
// 128-row Q tile per work unit, used at head dim 256, on sm_103a.  (The
// template also compiles for d = 128, where it measured slower than the
// two-Q-tile kernel: 1123 against 1524 TFLOP/s at B4 H16 N4096 when both
// used the shift of 8.)
//
// What it computes is the FP8 forward of fa_fwd_kernel.cuh ("FlashAttention-3
// on Hopper", sec. 6.3: e4m3 operands with one FP32 scale per 128-row tile;
// "03 FA3", sec. 4: the exponent of P shifted so that P uses the e4m3
// range): for each row, S_j = (alpha log2 e) q_s k_s (Q K_j^T) in log2
// units, P'_j = 2^(S_j - r + c) (v_j / v_max) rounded to e4m3, O += P'_j V_j,
// the row sum l counts 2^(S_j - r + c) without the V factor, and finally
// O = acc v_max / l, LSE = (r - c + log2 l) ln 2.  The reference r moves
// only when a tile's row max exceeds it by more than tau (conditional
// rescale, "FlashAttention v1-v4", FA4), so P' <= 2^(c + tau); here c = 4
// and tau = 4.8 (2^8.8 < 448, the largest e4m3 value).  The pages' shift of
// 8 with tau = 0.8 meets the same bound, but on the outlier inputs a warp
// then rescales its O rows on 31-63 % of key tiles, at ~2000 cycles each;
// with c = 4 that falls to about a sixth, and the terms of P' that lose
// precision (subnormal e4m3) are those below 2^-10 of the reference.
//
// Why a kernel of its own: at d = 256 the O accumulator of one Q tile takes
// 256 of the 512 TMEM columns, so the two-Q-tile schedule does not fit; and
// at d = 256 each exponential carries twice the tensor work of d = 128, which
// is where FP8 pays ("FlashAttention-3 on Hopper", sec. 6.5: the FP8 peak is
// reached at head dim 256).  Layout:
//   * TMEM: S0 [0,128), S1 [128,256) double-buffered FP32 scores of 128-key
//     tiles (P' as e4m3, 32 columns, overlays the first columns of its S
//     buffer), O [256,256+d);
//   * shared memory: two Q slots (e4m3; the next unit's Q loads while this
//     unit runs) and a ring of K/V tiles (5 stages of 32 KB at d = 256, 10
//     of 16 KB at d = 128), all in TMA's 128-byte swizzle (d / 128 column
//     chunks of 128 bytes per row);
//   * MMAs (kind::f8f6f4, FP32 accumulate): S[t%2] = Q K_t^T (both operands
//     in shared memory), O += P'[(t-1)%2] V_(t-1) (P' from TMEM, V as an
//     MN-major operand); per step the order is QK(t), PV(t-1), so the score
//     tile of step t+1 is computed while the softmax of step t runs.
// Warps: 0-3 softmax (thread = row = TMEM lane; also the epilogue), 4 TMA
// producer (one lane), 5 MMA issuer (converged warp, elect.sync issue).
// The softmax publishes P'(t) without waiting for PV(t-1) unless its rows'
// reference moved (the O correction needs PV(t-1) complete); it consumes
// every PV-done phase in order either way.  PV(t) completes on barrier
// PV_DONE[t % 2], so the next phase of a barrier needs P'(t+2), which the
// softmax publishes only after it has consumed PV(t): no barrier can run two
// phases ahead of its waiter.  Every mbarrier wait is bounded.
#pragma once

#include "fa_device.cuh"
#include "fa_fwd_kernel.cuh"   // FwdArgs

namespace fa {

template <int D_, bool kCausal>
struct Fp8Fwd1qCfg {
    static constexpr int D = D_;
    static_assert(D == 128 || D == 256, "head dim");
    static constexpr int BM = 128, BN = 128;
    static constexpr int NCH = D / 128;                     // 128-byte column chunks
    static constexpr uint32_t CHUNK = 128u * 128u;          // 128 rows x 128 B
    static constexpr uint32_t TILE_BYTES = NCH * CHUNK;     // Q, K or V tile: 16 or 32 KB
    static constexpr int NQ = 2;
    static constexpr int NSTAGE = D == 256 ? 5 : 10;
    static constexpr int NTHREADS = 192;
    static constexpr int QK_STEPS = D / 32;                 // 32 bytes of K per MMA
    static constexpr int PV_KEYS = 32;                      // keys per PV MMA
    static constexpr int PV_STEPS = BN / PV_KEYS;

    static constexpr uint32_t Q_OFF = 0;
    static constexpr uint32_t KV_OFF = NQ * TILE_BYTES;
    static constexpr uint32_t BAR_OFF = KV_OFF + NSTAGE * TILE_BYTES;
    static constexpr int B_QFULL = 0, B_QEMPTY = NQ, B_KVFULL = 2 * NQ,
                         B_KVEMPTY = B_KVFULL + NSTAGE, B_SFULL = B_KVEMPTY + NSTAGE,
                         B_PFULL = B_SFULL + 2, B_PVDONE = B_PFULL + 2,
                         B_OEMPTY = B_PVDONE + 2, B_MMADONE = B_OEMPTY + 1,
                         // causal: the dynamic order's answers (see the kernel)
                         B_CLCFULL = B_MMADONE + 1, B_UNIT = B_CLCFULL + 4,
                         B_CLCEMPTY = B_UNIT + 4, NBAR = B_CLCEMPTY + 4;
    static constexpr int CLC_DEPTH = 4;
    static constexpr uint32_t MISC_OFF = BAR_OFF + NBAR * 8;
    static constexpr uint32_t CLC_OFF = (MISC_OFF + 16 + 15) & ~15u;   // 16-byte aligned
    static constexpr uint32_t UNIT_OFF = CLC_OFF + CLC_DEPTH * 16;
    static constexpr uint32_t SMEM_BYTES = UNIT_OFF + CLC_DEPTH * 4 + 1024;   // + align slack
    static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");

    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_O = 256;
    static_assert(COL_O + D <= TMEM_COLS, "TMEM budget");
    __host__ __device__ static constexpr uint32_t col_s(int b) { return b ? 128u : 0u; }

    static constexpr uint32_t IDESC_QK = idesc_e4m3(128, BN, false, false);
    static constexpr uint32_t IDESC_PV = idesc_e4m3(128, D, false, true);
    // exponent offset c and rescale threshold tau: P' <= 2^(c + tau) =
    // 2^8.8 < 448 (see the header)
    static constexpr float TAU = 4.8f;
    static constexpr float P_OFFSET = 4.0f;
};

// Work unit: one 128-row Q tile m of one (b, h); key tiles jhi-1 down to 0.
struct UnitF8 {
    int b, h, m, T;
};

template <bool kCausal>
__device__ __forceinline__ UnitF8 make_unit_f8(int u, const FwdArgs &a) {
    UnitF8 U;
    const int BH = a.B * a.H;
    int bh;
    if (kCausal) {            // the dynamic order of fa_fwd_kernel.cuh
        dynamic_order(u, BH, a.n_kv, a.chunk, U.m, bh);
    } else {                  // consecutive units share a head's K/V in L2
        U.m = u % a.n_kv;
        bh = u / a.n_kv;
    }
    U.b = bh / a.H;
    U.h = bh % a.H;
    U.T = kCausal ? U.m + 1 : a.n_kv;
    return U;
}

template <int D, bool kCausal>
__global__ void __launch_bounds__(192, 1)
fa_fwd_fp8_1q_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const FwdArgs a) {
    using C = Fp8Fwd1qCfg<D, kCausal>;
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
        for (int q = 0; q < C::NQ; ++q) {
            mbar_init(bar(C::B_QFULL + q), 1);
            mbar_init(bar(C::B_QEMPTY + q), 1);
        }
        for (int s = 0; s < C::NSTAGE; ++s) {
            mbar_init(bar(C::B_KVFULL + s), 1);
            mbar_init(bar(C::B_KVEMPTY + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(C::B_SFULL + b), 1);
            mbar_init(bar(C::B_PFULL + b), 4);
            mbar_init(bar(C::B_PVDONE + b), 1);
        }
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
            uint32_t qc = 0, qarmed = 0, qarmed_par = 0;
            bool ok = true;
            auto load_kv = [&](const CUtensorMap *tm, const UnitF8 &U, int j) -> bool {
                if (!mbar_wait(bar(C::B_KVEMPTY + slot), phase ^ 1, w, 2)) return false;
                mbar_arrive_expect_tx(bar(C::B_KVFULL + slot), C::TILE_BYTES);
#pragma unroll
                for (int c = 0; c < C::NCH; ++c)
                    tma_load_4d(tm, base + C::KV_OFF + slot * C::TILE_BYTES + c * C::CHUNK,
                                bar(C::B_KVFULL + slot), c * 128, U.h / a.group, j * C::BN, U.b);
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
                const UnitF8 U = make_unit_f8<kCausal>(u, a);
                const uint32_t qs = qc % C::NQ, qph = (qc / C::NQ) & 1u;
                ok = mbar_wait(bar(C::B_QEMPTY + qs), qph ^ 1u, w, 1);
                if (!ok) break;
                mbar_arrive_expect_tx(bar(C::B_QFULL + qs), C::TILE_BYTES);
#pragma unroll
                for (int c = 0; c < C::NCH; ++c)
                    tma_load_4d(&tm_q, base + C::Q_OFF + qs * C::TILE_BYTES + c * C::CHUNK,
                                bar(C::B_QFULL + qs), c * 128, U.h, U.m * 128, U.b);
                qarmed |= 1u << qs;
                qarmed_par = (qarmed_par & ~(1u << qs)) | (qph << qs);
                ++qc;
                // ring order = MMA consumption order: K(0), then K(t), V(t-1)
                // for t = 1..T-1, then V(T-1); step t is key tile T-1-t.
                ok = load_kv(&tm_k, U, U.T - 1);
                for (int t = 1; ok && t < U.T; ++t) {
                    ok = load_kv(&tm_k, U, U.T - 1 - t);
                    if (ok) ok = load_kv(&tm_v, U, U.T - t);
                }
                if (ok) ok = load_kv(&tm_v, U, 0);
            }
            // Let every copy this lane issued land before the CTA can exit.
            if (kCausal && clc_pending)
                mbar_wait_quiet(bar(C::B_CLCFULL + (kq - 1) % C::CLC_DEPTH),
                                ((kq - 1) / C::CLC_DEPTH) & 1u, 500000000ull);
            for (int s = 0; s < C::NSTAGE; ++s)
                if (armed & (1u << s))
                    mbar_wait_quiet(bar(C::B_KVFULL + s), (armed_par >> s) & 1u, 500000000ull);
            for (int q = 0; q < C::NQ; ++q)
                if (qarmed & (1u << q))
                    mbar_wait_quiet(bar(C::B_QFULL + q), (qarmed_par >> q) & 1u, 500000000ull);
        }
        __syncwarp();
    } else if (warp == 5) {
        // =================== MMA issuer (whole warp, elected lane issues) ===================
        WaitCtx w{abort_flag, a.status, kRoleMma};
        uint32_t slot = 0, phase = 0, qc = 0;
        uint32_t pph0 = 0, pph1 = 0, un = 0;
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
            const UnitF8 U = make_unit_f8<kCausal>(u, a);
            const uint32_t qs = qc % C::NQ, qph = (qc / C::NQ) & 1u;
            ++qc;
            ok = mbar_wait_warp(bar(C::B_QFULL + qs), qph, w, 30);
            if (!ok) break;
            const uint64_t qd = smem_desc_sw128(base + C::Q_OFF + qs * C::TILE_BYTES, 16u, 1024u);
            for (int t = 0; t <= U.T && ok; ++t) {
                if (t < U.T) {
                    // ---- S[t%2] = Q K_t^T ----
                    uint32_t ks, kp;
                    next_slot(ks, kp);
                    ok = mbar_wait_warp(bar(C::B_KVFULL + ks), kp, w, 31);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t kd = smem_desc_sw128(base + C::KV_OFF + ks * C::TILE_BYTES, 16u, 1024u);
                    const uint32_t sb = t & 1;
#pragma unroll
                    for (int kk = 0; kk < C::QK_STEPS; ++kk) {
                        const uint32_t off = ((kk >> 2) * C::CHUNK + (kk & 3) * 32u) >> 4;
                        mma_ss_f8_elect(tbase + C::col_s(sb), qd + off, kd + off, C::IDESC_QK,
                                        kk > 0 ? 1u : 0u);
                    }
                    mma_commit_elect(bar(C::B_SFULL + sb));
                    mma_commit_elect(bar(C::B_KVEMPTY + ks));
                    if (t == U.T - 1) mma_commit_elect(bar(C::B_QEMPTY + qs));
                }
                if (t >= 1) {
                    // ---- O += P'[(t-1)%2] V_(t-1) ----
                    uint32_t vs, vp;
                    next_slot(vs, vp);
                    const uint32_t pb = (t - 1) & 1;
                    ok = mbar_wait_warp(bar(C::B_KVFULL + vs), vp, w, 32);
                    if (ok && t == 1) ok = mbar_wait_warp(bar(C::B_OEMPTY), (un & 1) ^ 1, w, 33);
                    if (ok) ok = mbar_wait_warp(bar(C::B_PFULL + pb), pb ? pph1 : pph0, w, 34);
                    if (!ok) break;
                    if (pb) pph1 ^= 1; else pph0 ^= 1;
                    tc_fence_after();
                    const uint64_t vd = smem_desc_sw128(base + C::KV_OFF + vs * C::TILE_BYTES,
                                                        C::CHUNK, 1024u);
#pragma unroll
                    for (int kk = 0; kk < C::PV_STEPS; ++kk)
                        mma_ts_f8_elect(tbase + C::COL_O, tbase + C::col_s(pb) + kk * 8u,
                                        vd + ((kk * C::PV_KEYS * 128u) >> 4), C::IDESC_PV,
                                        (t > 1 || kk > 0) ? 1u : 0u);
                    mma_commit_elect(bar(C::B_PVDONE + pb));
                    mma_commit_elect(bar(C::B_KVEMPTY + vs));
                }
            }
            ++un;
        }
        // Drain: every issued MMA completes before TMEM is released.
        mma_commit_elect(bar(C::B_MMADONE));
        mbar_wait_quiet(bar(C::B_MMADONE), 0, 500000000ull);
        __syncwarp();
    } else {
        // =================== softmax group (warps 0-3) ===================
        const int row = tid;                                     // TMEM lane == tile row
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        const uint32_t tO = tbase + lane_off + C::COL_O;
        WaitCtx w{abort_flag, a.status, kRoleSoftmax0};
        const float sl2 = a.scale_log2;
        uint32_t sph0 = 0, sph1 = 0, pvph0 = 0, pvph1 = 0;
        // consumes the completion phase of PV(t) (barrier PV_DONE[t % 2])
        auto wait_pv = [&](const int t, const uint32_t where) -> bool {
            const uint32_t b = t & 1;
            if (!mbar_wait(bar(C::B_PVDONE + b), b ? pvph1 : pvph0, w, where)) return false;
            if (b) pvph1 ^= 1; else pvph0 ^= 1;
            return true;
        };
        bool ok = true;
        bool pending_epi = false;
        UnitF8 P{};                      // the unit whose epilogue is pending
        float P_le = 0.f, P_r = -INFINITY, P_vmax = 1.f;

        // O of unit P is final once its last PV, PV(T-1), completed.
        auto epilogue = [&]() -> bool {
            if (!wait_pv(P.T - 1, 41)) return false;
            if (__any_sync(0xffffffffu, *abort_flag != 0u)) return false;
            tc_fence_after();
            const bool live = P_le > 0.f;
            const float inv = live ? P_vmax / P_le : 0.f;
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
                    pk[i] = pack2<true>(__uint_as_float(ov[2 * i]) * inv,
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
                const float lse2 = live ? P_r - C::P_OFFSET + log2f(P_le) : -INFINITY;
                a.lse[(static_cast<size_t>(P.b) * a.H + P.h) * a.N + grow] =
                    lse2 * 0.69314718055994530942f;
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
            const UnitF8 U = make_unit_f8<kCausal>(u, a);
            // The Q tile's scale and the largest V scale of the head (the
            // per-tile V scales are folded into P' relative to it).
            // Q scales per query head, K and V scales per K/V head
            const size_t sbase = (static_cast<size_t>(U.b) * a.H + U.h) * a.n_kv;
            const size_t kvbase = (static_cast<size_t>(U.b) * (a.H / a.group) + U.h / a.group) * a.n_kv;
            const float qsc = a.q_scale[sbase + U.m];
            float vm = 0.f;
            for (int jj = lane; jj < a.n_kv; jj += 32) vm = fmaxf(vm, a.v_scale[kvbase + jj]);
#pragma unroll
            for (int m = 16; m > 0; m >>= 1) vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, m));
            const float vmax = vm;
            // Per key tile: the score scale to log2 units with the q and k
            // tile scales ("FlashAttention-3 on Hopper", sec. 6.3), the
            // exponent offset c + log2(v_j / v_max) that carries the V tile
            // scale, and v_max / v_j for the row sum.  The next tile's scales
            // are loaded at the top of a tile (they land during the wait for
            // S) and turned into its constants after this tile's row sum:
            // neither sits on the path from S to P'.
            float ks_n, vs_n, sc_n, voff_n, ivr_n;
            auto tile_load = [&](const int j) __attribute__((always_inline)) {
                ks_n = a.k_scale[kvbase + j];
                vs_n = a.v_scale[kvbase + j];
            };
            auto tile_consts = [&]() __attribute__((always_inline)) {
                sc_n = sl2 * qsc * ks_n;
                voff_n = C::P_OFFSET + log2f(vs_n / vmax);
                ivr_n = vmax / vs_n;
            };
            tile_load(U.T - 1);
            tile_consts();
            // ---- epilogue of the previous unit, overlapped with this unit's
            //      first score tile ----
            if (pending_epi) {
                ok = epilogue();
                if (__any_sync(0xffffffffu, !ok)) { ok = false; break; }
                pending_epi = false;
            }
            float r = -INFINITY, le = 0.f;
            for (int t = 0; t < U.T; ++t) {
                const int j = U.T - 1 - t;
                const float sc = sc_n, voff = voff_n, ivr = ivr_n;
                if (t + 1 < U.T) tile_load(j - 1);
                const uint32_t sb = t & 1;
                ok = mbar_wait(bar(C::B_SFULL + sb), sb ? sph1 : sph0, w, 42);
                if (__any_sync(0xffffffffu, !ok)) { ok = false; break; }
                if (sb) sph1 ^= 1; else sph0 ^= 1;
                tc_fence_after();
                const uint32_t tS = tbase + lane_off + C::col_s(sb);
                uint32_t s[128];
                float *sf = reinterpret_cast<float *>(s);
                tmem_ld32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
                tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
                tmem_ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(&s[64]));
                tmem_ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(&s[96]));
                tmem_ld_wait();
                // ---- masks: sequence tail and causal diagonal ----
                int lim = 128;
                if (j == a.n_kv - 1) lim = min(lim, a.N - j * 128);
                if (kCausal && j == U.m) lim = min(lim, row + 1);
                if (lim < 128) {
#pragma unroll
                    for (int c = 0; c < 128; ++c) if (c >= lim) sf[c] = -INFINITY;
                }
                // ---- the row max first: e4m3 saturates above 448 ----
                float m0 = sf[0], m1 = sf[1], m2 = sf[2], m3 = sf[3];
#pragma unroll
                for (int c = 4; c < 128; c += 8) {
                    m0 = max3(m0, sf[c + 0], sf[c + 4]);
                    m1 = max3(m1, sf[c + 1], sf[c + 5]);
                    m2 = max3(m2, sf[c + 2], sf[c + 6]);
                    m3 = max3(m3, sf[c + 3], sf[c + 7]);
                }
                const float bnew = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3)) * sc;   // -inf stays -inf
                float rn = r, corr = 1.f;
                if (r == -INFINITY) rn = bnew;
                else { rn = (bnew > r + C::TAU) ? bnew : r; corr = ex2_approx(r - rn); }
                const bool need = (r != -INFINITY) && (rn != r);
                const float rs = (rn == -INFINITY) ? 0.f : rn;
                const float2 c2 = make_float2(sc, sc);
                const float2 nr2 = make_float2(voff - rs, voff - rs);
                float2 e_a = make_float2(0.f, 0.f), e_b = e_a;
                uint32_t p[32];
                // ---- P' = 2^(x - r + c) (v_j / v_max) as e4m3 ----
#pragma unroll
                for (int c = 0; c < 128; c += 4) {
                    const float2 x01 = __ffma2_rn(make_float2(sf[c + 0], sf[c + 1]), c2, nr2);
                    const float2 x23 = __ffma2_rn(make_float2(sf[c + 2], sf[c + 3]), c2, nr2);
                    const float2 e01 = make_float2(ex2_approx(x01.x), ex2_approx(x01.y));
                    const float2 e23 = make_float2(ex2_approx(x23.x), ex2_approx(x23.y));
                    p[c / 4] = pack4_e4m3(e01.x, e01.y, e23.x, e23.y);
                    e_a = __fadd2_rn(e_a, e01);
                    e_b = __fadd2_rn(e_b, e23);
                }
                tmem_st32(tS + 0, p);
                // ---- O correction: PV(t-1) must have completed first ----
                const bool fix = __any_sync(0xffffffffu, need);
                bool waited = false;
                if (t > 0 && fix) {
                    ok = wait_pv(t - 1, 43);
                    if (__any_sync(0xffffffffu, !ok)) { ok = false; break; }
                    waited = true;
                    tc_fence_after();
                }
                if (fix) {
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
                // every PV-done phase is consumed once, in order
                if (t > 0 && !waited) {
                    ok = wait_pv(t - 1, 44);
                    if (__any_sync(0xffffffffu, !ok)) { ok = false; break; }
                }
                // the row sum counts 2^(x - r + c) without the V factor
                le = __fmaf_rn(le, corr, ((e_a.x + e_a.y) + (e_b.x + e_b.y)) * ivr);
                r = rn;
                if (t + 1 < U.T) tile_consts();
            }
            if (!ok) break;
            P = U;
            P_le = le;
            P_r = r;
            P_vmax = vmax;
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
