// fa_fwd_kernel.cuh -- exact attention forward on sm_103a (tcgen05 + TMA).
//
// What it computes ("FlashAttention-3 on Hopper", sec. 4.1-4.7): for every
// (batch b, head h) and query row i,
//     O_i = sum_j softmax_j(alpha q_i . k_j) v_j,   LSE_i = log sum_j exp(.)
// over visible keys j (causal: j <= i), tile by tile with an online softmax
// so no N x N matrix is stored.
//
// How (the Blackwell forward schedule of "FlashAttention v1-v4", FA4
// sections "TMEM", "forward schedule: two Q tiles, two softmax groups" and
// "conditional rescale", re-planned for GB300):
//   * A work unit is a pair of 128-row Q tiles (tile L = 2p, tile H = 2p+1)
//     of one (b, h); both share one stream of 128-key K/V tiles, visited in
//     descending order so that the masked tiles (sequence tail, causal
//     diagonal) come first ("FlashAttention-3 on Hopper", sec. 4.7).
//     Persistent grid, one CTA per SM, except for causal units, which are
//     scheduled dynamically (make_unit): one CTA per unit, running CTAs
//     taking over those not yet started.
//   * 384 threads; warpgroup 2 (warps 8-11) gives registers to the two
//     softmax warpgroups with setmaxnreg.  Warps 10-11 are spare.
//   * Warp 8 (one lane) is the TMA producer: Q_L/Q_H once per unit into
//     three rotating Q slots (the next unit's first Q tile loads while the
//     current unit runs), then K_j and V_j into a ring of shared-memory
//     stages guarded by full/empty mbarriers ("FlashAttention-3 on Hopper",
//     sec. 4.3.1).
//   * Warp 9 (one lane) issues every tcgen05.mma: S_X = Q_X K_j^T into
//     TMEM, O_X += P_X V_j with P_X read from TMEM (TS form).  Per step the
//     order is PV_L(j+1), QK_L(j), PV_H(j+1), QK_H(j), so each softmax group
//     has the other tile's two GEMMs to hide behind.
//   * Warps 0-3 / 4-7 are the softmax groups for tiles L / H: thread t owns
//     row t (TMEM lane t), reads its 128 scores with tcgen05.ld, masks,
//     takes the row max, applies the conditional-rescale rule with threshold
//     tau = 8 (log2 units), evaluates exp2 on MUFU, rounds P to bf16/fp16,
//     accumulates the row sum of those rounded values in FP32, writes P back
//     over its S columns with tcgen05.st,
//     and rescales its O row in TMEM when the reference point moved.  After
//     the last tile it normalises O by 1/l and stores O (32-byte stores, so
//     each store fills whole sectors of its row) and LSE.
//   * TMEM (512 columns): S_L [0,128), S_H [128,256), O_L [256,256+D),
//     O_H [256+D, 256+2D); P_X (64 columns of packed pairs) overlays the
//     first half of S_X.
// Every mbarrier wait is bounded (fa_device.cuh).
#pragma once

#include "fa_device.cuh"

namespace fa {

struct FwdArgs {
    void *o;             // [B][N][H][D]
    float *lse;          // [B][H][N] or nullptr
    uint32_t *status;    // device status word (4 x u32)
    int B, H, N;
    int n_kv;            // ceil(N / 128) key tiles
    int n_pairs;         // ceil(ceil(N / 128) / 2) Q-tile pairs per head
    int n_units;         // B * H * n_pairs
    int group;           // query heads per K/V head (1: one K/V head per query head)
    // Split key ranges (d <= 128, 16-bit): n_splits >= 1; with o_part set,
    // split s of a unit writes its partial O (FP32, normalised by its own
    // row sum) to o_part [S][B][N][H][D] and its LSE to lse_part [S][B][H][N]
    // instead of O and LSE.  Causal units without splits or packing take
    // the dynamic order of make_unit instead, whose groups hold chunk heads
    // (>= 1); the two never meet in one launch.
    union {
        int n_splits;
        int chunk;
    };
    float *o_part, *lse_part;
    float scale_log2;    // alpha * log2(e)
    // Score and mask variants (kExt instantiations only).  Key j is hidden
    // from query i when j > i + wr (wr >= 0) or j < i - wl (wl >= 0); -1 is
    // no bound.  Softcap c: each score s becomes c tanh(alpha s / c), formed
    // as sc_post * tanh(sc_pre * s) with sc_pre = alpha / c and
    // sc_post = c log2(e) (sc_pre = 0: no softcap).  sinks: one logit per
    // query head, added to every row's softmax denominator, or null.
    int wl, wr;
    float sc_pre, sc_post;
    const float *sinks;
    // FP8 only: one FP32 scale per 128-row tile of each head, [B][H][n_kv]
    const float *q_scale, *k_scale, *v_scale;
};

// kFP8: Q/K/V are e4m3 codes with per-tile scales (kind::f8f6f4 MMAs), O is
// bf16.  Otherwise Q/K/V/O are bf16 (kBF16) or fp16.
template <int D, bool kCausal, bool kBF16, bool kFP8 = false>
struct FwdCfg {
    static_assert(D == 64 || D == 128, "head dim");
    static_assert(!kFP8 || (D == 128 && kBF16), "FP8 path: d = 128, bf16 output");
    static constexpr int ESZ = kFP8 ? 1 : 2;            // bytes per Q/K/V element
    static constexpr int BM = 128;                      // query rows per tile
    static constexpr int BN = 128;                      // keys per tile
    static constexpr int NCH = D * ESZ / 128;           // 128-byte column chunks
    static constexpr uint32_t CHUNK_BYTES = 128u * 128u;  // 128 rows x 128 B
    static constexpr uint32_t TILE_BYTES = NCH * CHUNK_BYTES;
    // K/V ring stages and Q slots.  Three Q slots rotate over the units'
    // tiles, so the next unit's first Q tile loads while this unit still
    // runs (two slots would make it wait for this unit's last QK).
    static constexpr int NSTAGE = (kFP8 || D == 64) ? 8 : 4;
    static constexpr int NQ = 3;
    static constexpr int QK_STEPS = D * ESZ / 32;       // 32 bytes of K per MMA
    static constexpr int PV_KEYS = 32 / ESZ;            // keys per PV MMA
    static constexpr int PV_STEPS = BN / PV_KEYS;
    static constexpr int P_COLS = BN * ESZ / 4;         // TMEM columns of P
    // 12 warps: 0-7 softmax groups, 8 TMA producer, 9 MMA issuer, 10-11
    // spare.  Launch budget 384 x 168 registers; warpgroup 2 shrinks to
    // REGS_LOW so the two softmax warpgroups can grow to REGS_HIGH:
    // 128*REGS_LOW + 256*REGS_HIGH <= 384*168.
    static constexpr int NTHREADS = 384;
    static constexpr uint32_t REGS_LOW = 96, REGS_HIGH = 200;
    static_assert(128 * REGS_LOW + 256 * REGS_HIGH <= 384 * 168, "register budget");

    // d = 64: the row sum of the rounded P comes from the tensor core, as a
    // 16-column accumulator L_X += P_X 1 next to O_X (TMEM has room at d = 64;
    // at d = 128 S and O fill it), which takes 128 additions per tile off
    // the softmax warps.
    static constexpr bool kLMMA = D == 64 && !kFP8;
    // shared memory map (offsets from a 1024-B aligned base); ONES: a 2 KB
    // block of 16-bit ones, the B operand of the L product (every element
    // it reads is 1, so one descriptor serves every key step)
    static constexpr uint32_t Q_OFF = 0;
    static constexpr uint32_t KV_OFF = NQ * TILE_BYTES;
    static constexpr uint32_t ONES_OFF = KV_OFF + NSTAGE * TILE_BYTES;
    static constexpr uint32_t BAR_OFF = ONES_OFF + (kLMMA ? 2048u : 0u);
    // barrier indices
    static constexpr int B_QFULL = 0, B_QEMPTY = NQ, B_KVFULL = 2 * NQ,
                         B_KVEMPTY = 2 * NQ + NSTAGE, B_SFULL = 2 * NQ + 2 * NSTAGE,
                         B_PFULL = B_SFULL + 2, B_OFULL = B_PFULL + 2,
                         B_OEMPTY = B_OFULL + 2, B_MMADONE = B_OEMPTY + 2,
                         // dynamic order: the hardware's answer for the next
                         // unit landed, its block index published, slot free
                         B_CLCFULL = B_MMADONE + 1, B_UNIT = B_CLCFULL + 4,
                         B_CLCEMPTY = B_UNIT + 4, NBAR = B_CLCEMPTY + 4;
    static constexpr int CLC_DEPTH = 4;          // units the producer may run ahead
    static constexpr uint32_t MISC_OFF = BAR_OFF + NBAR * 8;
    // 16 B per answer, 16-byte aligned (the answer's store and its 128-bit load)
    static constexpr uint32_t CLC_OFF = (MISC_OFF + 16 + 15) & ~15u;
    static_assert(CLC_OFF % 16 == 0, "cluster launch control answers: 16-byte aligned");
    static constexpr uint32_t UNIT_OFF = CLC_OFF + CLC_DEPTH * 16;   // int per answer
    static constexpr uint32_t SMEM_BYTES = UNIT_OFF + CLC_DEPTH * 4 + 1024;   // + align slack
    static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");

    // TMEM columns
    static constexpr uint32_t TMEM_COLS = 512;
    __host__ __device__ static constexpr uint32_t col_s(int x) { return x ? 128u : 0u; }
    __host__ __device__ static constexpr uint32_t col_o(int x) { return 256u + (x ? D : 0u); }
    __host__ __device__ static constexpr uint32_t col_l(int x) { return 256u + 2u * D + (x ? 16u : 0u); }
    static_assert(!kLMMA || col_l(1) + 16 <= TMEM_COLS, "TMEM budget of L");

    static constexpr uint32_t IDESC_QK =
        kFP8 ? idesc_e4m3(128, 128, false, false) : idesc_f16(128, 128, kBF16, false, false);
    static constexpr uint32_t IDESC_PV =
        kFP8 ? idesc_e4m3(128, D, false, true) : idesc_f16(128, D, kBF16, false, true);
    static constexpr uint32_t IDESC_L = idesc_f16(128, 16, kBF16, false, true);
    // Conditional-rescale threshold (log2 units).  16-bit P: tau = 8, so
    // P <= 2^8.  FP8 P ("03 FA3", sec. 4, Max_offset): the exponent is
    // shifted by c = 4 into the e4m3 range and tau = 4.8 keeps
    // P <= 2^8.8 < 448, the largest e4m3 value.  The pages' c = 8 leaves
    // tau = 0.8, and the O correction that a moved reference needs (done
    // before P is published) then runs on about half of the warp-steps of
    // the outlier inputs; c = 4 rescales a tenth as often, for 1.4 % more
    // RMSE (terms below 2^-10 of the reference become e4m3 subnormals).
    static constexpr float TAU = kFP8 ? 4.8f : 8.0f;
    static constexpr float P_OFFSET = kFP8 ? 4.0f : 0.0f;
    // 16-bit P is first formed against the current reference r and kept
    // when the tile's FP32 row sum is <= 2^16.  The sum bounds every term,
    // so a kept tile has P <= 2^16; a tile that fails has a term > 2^16/128
    // = 2^9 > 2^tau, so its row max grew by more than tau and r moves.
    static constexpr float KEEP_SUM = 65536.0f;
};

// The geometry of one work unit, identical in every role.
struct Unit {
    int b, h;
    int m[2];       // Q tile indices (L, H)
    bool act[2];    // tile takes part in this unit (real rows, keys in range)
    int T;          // key tiles visited: jhi-1 down to jhi-T
    int jhi;        // one past the unit's highest key tile
    int t0[2];      // first step at which tile X takes part (T if never)
    int t1[2];      // one past its last step (T unless a left window ends it)
    int s;          // split of the key range
};

// Visible keys [klo, khi) of query row i under the window (wl, wr); every
// row in [0, N) sees at least key i.  Written with min() so that no
// intermediate leaves [0, N] for any window value.
__device__ __forceinline__ int window_lo(int i, const FwdArgs &a) {
    return a.wl >= 0 ? i - min(a.wl, i) : 0;
}
__device__ __forceinline__ int window_hi(int i, const FwdArgs &a) {
    return a.wr >= 0 ? i + 1 + min(a.wr, a.N - 1 - i) : a.N;
}

// Units whose length falls with their index (longest-first orders).
template <bool kCausal, bool kExt>
__device__ __forceinline__ bool units_longest_first(const FwdArgs &a) {
    return kExt ? (a.wl < 0 && a.wr >= 0) : kCausal;
}

// kSplit: the key range is cut into a.n_splits parts (otherwise one part,
// folded away at compile time).  kExt: the key range of each Q tile comes
// from the window ("FlashAttention-3 on Hopper", sec. 4.7: local attention
// bounds the loop on both sides), so a tile may also leave the pair's
// descending key stream before its end.
// kPack (grouped heads, "PackGQA"): the a.group query heads of one K/V head
// share each Q tile -- tile row p holds query position m R + p / group of
// query head h group + p % group, R = 128 / group -- so units run over K/V
// heads (U.h is then the K/V head) and one K/V stream serves the whole
// group.  R divides 128, so a tile's positions never straddle a key tile.
// Causal units without splits or packing are taken in a dynamic order:
// each CTA asks the hardware for its next unit when it needs it (cluster
// launch control), so a CTA that finishes early takes more.  The order
// keeps a group of a.chunk heads together, longest pair first within the
// group, so the group's K/V stay in L2 while its units run; the shortest
// pair of every head (one or two key tiles) comes last, over all heads,
// so that the CTAs finish together.
template <bool kCausal, bool kSplit, bool kExt, bool kPack>
__device__ __forceinline__ constexpr bool dynamic_units() {
    return kCausal && !kSplit && !kExt && !kPack;
}

template <bool kCausal, bool kSplit, bool kExt = false, bool kPack = false>
__device__ __forceinline__ Unit make_unit(int u, const FwdArgs &a) {
    Unit U;
    const int HH = kPack ? a.H / a.group : a.H;    // heads the units run over
    const int BH = a.B * HH;
    const int S = kSplit ? a.n_splits : 1;
    U.s = kSplit ? u % S : 0;       // the splits of one pair are adjacent units
    if (kSplit) u /= S;
    int p, bh;
    // a right bound without a left one makes later pairs longer
    const bool lpt = units_longest_first<kCausal, kExt>(a);
    if (dynamic_units<kCausal, kSplit, kExt, kPack>()) {
        const int P1 = a.n_pairs - 1;              // pairs per head before the tail
        const int grouped = BH * P1;
        if (u < grouped) {
            const int g = u / (a.chunk * P1);
            const int r = u - g * a.chunk * P1;
            const int cg = min(a.chunk, BH - g * a.chunk);   // heads in this group
            p = P1 - r / cg;
            bh = g * a.chunk + r % cg;
        } else {
            p = 0;
            bh = u - grouped;
        }
    } else if (lpt) {       // longest-first: the last pairs of every head first
        p = a.n_pairs - 1 - u / BH;
        bh = u % BH;
    } else {                // consecutive units share a head's K/V in L2
        p = u % a.n_pairs;
        bh = u / a.n_pairs;
    }
    U.b = bh / HH;
    U.h = bh % HH;
    if constexpr (kExt) {
        int lo[2] = {0, 0}, hi[2] = {0, 0};
        for (int x = 0; x < 2; ++x) {
            U.m[x] = 2 * p + x;
            U.act[x] = U.m[x] * 128 < a.N;
            if (U.act[x]) {
                const int r0 = U.m[x] * 128, r1 = min(a.N, r0 + 128) - 1;
                const int klo = window_lo(r0, a), khi = window_hi(r1, a);
                lo[x] = klo >> 7;
                hi[x] = (khi >> 7) + ((khi & 127) != 0);
            }
        }
        // tile H's range ends at or above tile L's and starts at or above
        // it, and the two ranges touch (each row sees its diagonal key)
        U.jhi = U.act[1] ? hi[1] : hi[0];
        U.T = U.jhi - lo[0];
        for (int x = 0; x < 2; ++x) {
            U.t0[x] = U.act[x] ? U.jhi - hi[x] : U.T;
            U.t1[x] = U.act[x] ? U.jhi - lo[x] : U.T;
        }
        return U;
    }
    int hi[2];
    for (int x = 0; x < 2; ++x) {
        U.m[x] = 2 * p + x;
        if constexpr (kPack) {
            const int q0 = U.m[x] * (128 / a.group);          // first position of the tile
            U.act[x] = q0 < a.N;
            hi[x] = U.act[x] ? (kCausal ? min(a.n_kv, (q0 >> 7) + 1) : a.n_kv) : 0;
        } else {
            U.act[x] = U.m[x] * 128 < a.N;
            hi[x] = U.act[x] ? (kCausal ? min(a.n_kv, U.m[x] + 1) : a.n_kv) : 0;
        }
    }
    // split s of the pair's key range [0, Tf): tiles [Tf s / S, Tf (s+1) / S)
    const int Tf = max(hi[0], hi[1]);
    const int lo = kSplit ? Tf * U.s / S : 0;
    U.jhi = kSplit ? Tf * (U.s + 1) / S : Tf;
    U.T = U.jhi - lo;
    for (int x = 0; x < 2; ++x) {
        const int cnt = max(0, min(hi[x], U.jhi) - lo);
        U.act[x] = cnt > 0;
        U.t0[x] = U.T - cnt;
        U.t1[x] = U.T;
    }
    return U;
}

// kVar: the score and mask variants of FwdArgs -- 1: window and sinks,
// 2: window, sinks and softcap; kCausal is then unused (the causal mask is
// the window (-1, 0)).
template <int D, bool kCausal, bool kBF16, bool kFP8 = false, bool kSplit = false,
          int kVar = 0, bool kPack = false>
__global__ void __launch_bounds__(384, 1)
fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
              const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const FwdArgs a) {
    using C = FwdCfg<D, kCausal, kBF16, kFP8>;
    constexpr bool kExt = kVar != 0;
    constexpr bool kCap = kVar == 2;
    static_assert(!kExt || (!kFP8 && !kSplit && !kCausal), "variants: 16-bit, one split");
    static_assert(!kPack || (!kExt && !kFP8 && !kSplit), "packed heads: plain or causal, 16-bit");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const bool snake = units_longest_first<kCausal, kExt>(a);   // unit order (unit_stride0)
    // Dynamic order: the grid has one CTA per unit; a CTA starts with its
    // own unit and then takes the units of CTAs it cancels before they
    // launch.  The producer asks for the next unit once it has issued the
    // loads of the current one; the k-th answer goes to slot k % CLC_DEPTH,
    // the producer publishes its block index there (-1: none left), and the
    // MMA warp and the 8 softmax warps read it and release the slot.
    // Static order: the persistent stride walk.
    volatile int *unit_slot = reinterpret_cast<volatile int *>(gbase + C::UNIT_OFF);
    constexpr bool kDyn = dynamic_units<kCausal, kSplit, kExt, kPack>();

    auto bar = [&](int i) -> uint32_t { return base + C::BAR_OFF + 8u * i; };
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(gbase + C::MISC_OFF);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(gbase + C::MISC_OFF + 4);

    // ---- prologue: TMEM allocation (warp 9) and barrier init (thread 0) ----
    if (warp == 9) tmem_alloc(base + C::MISC_OFF, C::TMEM_COLS);
    if (tid == 0) {
        *abort_flag = 0u;
        for (int q = 0; q < C::NQ; ++q) {
            mbar_init(bar(C::B_QFULL + q), 1);
            mbar_init(bar(C::B_QEMPTY + q), 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(bar(C::B_SFULL + x), 1);
            mbar_init(bar(C::B_PFULL + x), 4);
            mbar_init(bar(C::B_OFULL + x), 1);
            mbar_init(bar(C::B_OEMPTY + x), 4);
        }
        for (int s = 0; s < C::NSTAGE; ++s) {
            mbar_init(bar(C::B_KVFULL + s), 1);
            mbar_init(bar(C::B_KVEMPTY + s), 1);
        }
        mbar_init(bar(C::B_MMADONE), 1);
        for (int q = 0; kDyn && q < C::CLC_DEPTH; ++q) {
            mbar_init(bar(C::B_CLCFULL + q), 1);
            mbar_init(bar(C::B_UNIT + q), 1);
            mbar_init(bar(C::B_CLCEMPTY + q), 9);
        }
        fence_barrier_init();
    }
    if constexpr (C::kLMMA) {
        // the ones block (2048 B of 16-bit 1.0), written here and read by the
        // tensor core: made visible to the async proxy before the barrier
        const uint32_t one2 = kBF16 ? 0x3F803F80u : 0x3C003C00u;
        for (int i = tid; i < 512; i += C::NTHREADS)
            reinterpret_cast<uint32_t *>(gbase + C::ONES_OFF)[i] = one2;
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;

    if (warp >= 8) {
      // Warpgroup 2 gives up registers first; each branch below starts with
      // its warpgroup's setmaxnreg so the register budget of every role is
      // known on every path into it.
      regs_shrink<C::REGS_LOW>();
      if (warp == 8) {
        // =================== TMA producer (one lane) ===================
        if (lane == 0) {
            WaitCtx w{abort_flag, a.status, kRoleProducer};
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            uint32_t qc = 0;                        // Q loads issued (slot qc % NQ)
            uint32_t qarmed = 0, qarmed_par = 0;    // per Q slot: ever loaded / parity
            uint32_t slot = 0, phase = 0;
            uint32_t armed = 0, armed_par = 0;      // per-slot: ever armed / parity
            bool ok = true;
            // Tile x of U into the next Q slot, once the slot's previous
            // tile has had its last QK.
            auto load_q = [&](const int x, const Unit &U) __attribute__((always_inline)) -> bool {
                const uint32_t qs = qc % C::NQ, qph = (qc / C::NQ) & 1u;
                if (!mbar_wait(bar(C::B_QEMPTY + qs), qph ^ 1u, w, 1)) return false;
                mbar_arrive_expect_tx(bar(C::B_QFULL + qs), C::TILE_BYTES);
#pragma unroll
                for (int c = 0; c < C::NCH; ++c)
                    tma_load_4d(&tm_q, base + C::Q_OFF + qs * C::TILE_BYTES + c * C::CHUNK_BYTES,
                                bar(C::B_QFULL + qs), c * (128 / C::ESZ),
                                kPack ? U.h * a.group : U.h,                 // packed: box of group heads
                                kPack ? U.m[x] * (128 / a.group) : U.m[x] * 128, U.b);
                qarmed |= 1u << qs;
                qarmed_par = (qarmed_par & ~(1u << qs)) | (qph << qs);
                ++qc;
                return true;
            };
            // dynamic order: the k-th request (k = 0, 1, ...) uses slot
            // k % CLC_DEPTH, once its readers have released answer k - CLC_DEPTH
            uint32_t kq = 0;                        // requests issued
            bool clc_pending = false;               // a request without its answer
            auto next_dyn = [&]() __attribute__((always_inline)) -> int {
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
            for (int u = blockIdx.x, st = unit_stride0(snake); ok && (!kDyn || u >= 0) && u < a.n_units;
                     u = kDyn ? next_dyn() : u + st, st = 2 * static_cast<int>(gridDim.x) - st) {
                const Unit U = make_unit<kCausal, kSplit, kExt, kPack>(u, a);
                if (U.act[0]) ok = ok && load_q(0, U);
                if (U.act[1]) ok = ok && load_q(1, U);
                const int hk = kPack ? U.h : U.h / a.group;   // K/V head of this query head
                for (int t = 0; t < U.T && ok; ++t) {
                    const int j = U.jhi - 1 - t;
                    for (int kv = 0; kv < 2; ++kv) {
                        ok = mbar_wait(bar(C::B_KVEMPTY + slot), phase ^ 1, w, 2);
                        if (!ok) break;
                        mbar_arrive_expect_tx(bar(C::B_KVFULL + slot), C::TILE_BYTES);
                        const CUtensorMap *tm = kv ? &tm_v : &tm_k;
                        for (int c = 0; c < C::NCH; ++c)
                            tma_load_4d(tm, base + C::KV_OFF + slot * C::TILE_BYTES + c * C::CHUNK_BYTES,
                                        bar(C::B_KVFULL + slot), c * (128 / C::ESZ), hk, j * 128, U.b);
                        armed |= 1u << slot;
                        armed_par = (armed_par & ~(1u << slot)) | (phase << slot);
                        if (++slot == C::NSTAGE) { slot = 0; phase ^= 1; }
                    }
                }
            }
            // Let every copy this lane issued land before the CTA can exit.
            if (kDyn && clc_pending)
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
    } else if (warp == 9) {
        // =================== MMA issuer (whole warp, one elected lane issues) ===================
        {
            WaitCtx w{abort_flag, a.status, kRoleMma};
            uint32_t qc = 0;                        // Q slots in the producer's order
            int un0 = 0, un1 = 0;
            uint32_t pph0 = 0, pph1 = 0;
            uint32_t slot = 0, phase = 0;
            bool ok = true;
            uint32_t kq = 0;                        // dynamic order: answers read
            auto next_dyn = [&]() __attribute__((always_inline)) -> int {
                if (!ok) return -1;
                const uint32_t q = kq % C::CLC_DEPTH, ph = (kq / C::CLC_DEPTH) & 1u;
                ++kq;
                if (!mbar_wait_warp(bar(C::B_UNIT + q), ph, w, 15)) { ok = false; return -1; }
                const int nu = unit_slot[q];
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::B_CLCEMPTY + q));
                return nu;
            };
            for (int u = blockIdx.x, st = unit_stride0(snake); ok && (!kDyn || u >= 0) && u < a.n_units;
                     u = kDyn ? next_dyn() : u + st, st = 2 * static_cast<int>(gridDim.x) - st) {
                const Unit U = make_unit<kCausal, kSplit, kExt, kPack>(u, a);
                uint32_t qs0 = 0, qp0 = 0, qs1 = 0, qp1 = 0;   // Q slot and parity per tile
                if (U.act[0]) { qs0 = qc % C::NQ; qp0 = (qc / C::NQ) & 1u; ++qc; }
                if (U.act[1]) { qs1 = qc % C::NQ; qp1 = (qc / C::NQ) & 1u; ++qc; }
                for (int t = 0; t <= U.T && ok; ++t) {
                    const bool has_v = t > 0, has_k = t < U.T;
                    uint32_t vslot = 0, vph = 0, kslot = 0, kph = 0;
                    if (has_v) { vslot = slot; vph = phase; if (++slot == C::NSTAGE) { slot = 0; phase ^= 1; } }
                    if (has_k) { kslot = slot; kph = phase; if (++slot == C::NSTAGE) { slot = 0; phase ^= 1; } }
                    bool v_ready = false, k_ready = false;
                    // One Q tile's two GEMMs of this step; x is a literal at
                    // each call site, so every per-tile counter is a register.
                    auto step_x = [&](const int x, const int t0x, const int t1x, const uint32_t qs,
                                      const uint32_t qp, int &un,
                                      uint32_t &pph) __attribute__((always_inline)) -> bool {
                        // ---- O_x += P_x V_(t-1) ----
                        if (has_v && t - 1 >= t0x && (!kExt || t - 1 < t1x)) {
                            if (!v_ready) {
                                if (!mbar_wait_warp(bar(C::B_KVFULL + vslot), vph, w, 10)) return false;
                                v_ready = true;
                            }
                            if (t - 1 == t0x &&
                                !mbar_wait_warp(bar(C::B_OEMPTY + x), (un & 1) ^ 1, w, 11)) return false;
                            if (!mbar_wait_warp(bar(C::B_PFULL + x), pph, w, 12)) return false;
                            tc_fence_after();
                            const uint64_t vd = smem_desc_sw128(base + C::KV_OFF + vslot * C::TILE_BYTES,
                                                                C::CHUNK_BYTES, 1024u);
                            const uint32_t acc = (t - 1 > t0x) ? 1u : 0u;
#pragma unroll
                            for (int kk = 0; kk < C::PV_STEPS; ++kk) {
                                const uint64_t bd = vd + ((kk * C::PV_KEYS * 128u) >> 4);
                                if constexpr (kFP8)
                                    mma_ts_f8_elect(tbase + C::col_o(x), tbase + C::col_s(x) + kk * 8u,
                                                    bd, C::IDESC_PV, (acc | kk) ? 1u : 0u);
                                else
                                    mma_ts_f16_elect(tbase + C::col_o(x), tbase + C::col_s(x) + kk * 8u,
                                                     bd, C::IDESC_PV, (acc | kk) ? 1u : 0u);
                                if constexpr (C::kLMMA)     // L_X += P_X 1 (row sums of P)
                                    mma_ts_f16_elect(tbase + C::col_l(x), tbase + C::col_s(x) + kk * 8u,
                                                     smem_desc_sw128(base + C::ONES_OFF, 16u, 1024u),
                                                     C::IDESC_L, (acc | kk) ? 1u : 0u);
                            }
                            pph ^= 1;
                            if (t == t1x) mma_commit_elect(bar(C::B_OFULL + x));
                        }
                        // ---- S_x = Q_x K_t^T ----
                        if (has_k && t >= t0x && (!kExt || t < t1x)) {
                            if (!k_ready) {
                                if (!mbar_wait_warp(bar(C::B_KVFULL + kslot), kph, w, 13)) return false;
                                k_ready = true;
                            }
                            if (t == t0x &&
                                !mbar_wait_warp(bar(C::B_QFULL + qs), qp, w, 14)) return false;
                            tc_fence_after();
                            const uint64_t qd = smem_desc_sw128(base + C::Q_OFF + qs * C::TILE_BYTES, 16u, 1024u);
                            const uint64_t kd = smem_desc_sw128(base + C::KV_OFF + kslot * C::TILE_BYTES, 16u, 1024u);
#pragma unroll
                            for (int kk = 0; kk < C::QK_STEPS; ++kk) {
                                const uint32_t off = ((kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32u) >> 4;
                                if constexpr (kFP8)
                                    mma_ss_f8_elect(tbase + C::col_s(x), qd + off, kd + off,
                                                    C::IDESC_QK, kk > 0 ? 1u : 0u);
                                else
                                    mma_ss_f16_elect(tbase + C::col_s(x), qd + off, kd + off,
                                                     C::IDESC_QK, kk > 0 ? 1u : 0u);
                            }
                            mma_commit_elect(bar(C::B_SFULL + x));
                            if (t == t1x - 1) mma_commit_elect(bar(C::B_QEMPTY + qs));
                        }
                        return true;
                    };
                    ok = step_x(0, U.t0[0], kExt ? U.t1[0] : U.T, qs0, qp0, un0, pph0) &&
                         step_x(1, U.t0[1], kExt ? U.t1[1] : U.T, qs1, qp1, un1, pph1);
                    if (!ok) break;
                    if (has_k) mma_commit_elect(bar(C::B_KVEMPTY + kslot));
                    if (has_v) mma_commit_elect(bar(C::B_KVEMPTY + vslot));
                }
                un0 += U.act[0] ? 1 : 0;
                un1 += U.act[1] ? 1 : 0;
            }
            // Drain: every issued MMA completes before TMEM is released.
            mma_commit_elect(bar(C::B_MMADONE));
            mbar_wait_quiet(bar(C::B_MMADONE), 0, 500000000ull);
        }
        __syncwarp();
      }
    } else {
        regs_grow<C::REGS_HIGH>();
        // =================== softmax group x (warps 4x .. 4x+3) ===================
        const int x = warp >> 2;
        const int row = tid & 127;                       // TMEM lane == tile row
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tbase + lane_off + C::col_s(x);
        const uint32_t tO = tbase + lane_off + C::col_o(x);
        const uint32_t tL = tbase + lane_off + (C::kLMMA ? C::col_l(x) : 0u);
        WaitCtx w{abort_flag, a.status, x ? kRoleSoftmax1 : kRoleSoftmax0};
        // With a softcap the scores reaching the softmax are tanh values in
        // [-1, 1], scaled to log2 units by c log2(e).
        const float sc_pre = kCap ? a.sc_pre : 0.f;
        const float sl2 = kCap ? a.sc_post : a.scale_log2;
        uint32_t sph = 0, oph = 0;
        // O rows are D * 2 (partials D * 4) bytes apart, a multiple of 32, so
        // 32-byte stores are aligned everywhere when the base is; the API
        // promises only 16 bytes, and 16-byte stores serve that case.
        const bool v8ok =
            ((reinterpret_cast<uintptr_t>(kSplit ? static_cast<const void *>(a.o_part) : a.o) & 31u) == 0);
        bool ok = true;
        uint32_t kq = 0;                            // dynamic order: answers read
        // (a failed wait leaves this loop by break, so ok holds here)
        auto next_dyn = [&]() __attribute__((always_inline)) -> int {
            const uint32_t q = kq % C::CLC_DEPTH, ph = (kq / C::CLC_DEPTH) & 1u;
            ++kq;
            ok = mbar_wait(bar(C::B_UNIT + q), ph, w, 23);
            if (__any_sync(0xffffffffu, !ok)) { ok = false; return -1; }
            const int nu = unit_slot[q];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_CLCEMPTY + q));
            return nu;
        };
        for (int u = blockIdx.x, st = unit_stride0(snake); ok && (!kDyn || u >= 0) && u < a.n_units;
                     u = kDyn ? next_dyn() : u + st, st = 2 * static_cast<int>(gridDim.x) - st) {
            const Unit U = make_unit<kCausal, kSplit, kExt, kPack>(u, a);
            const bool act = x ? U.act[1] : U.act[0];
            if (!act) continue;
            const int mt = x ? U.m[1] : U.m[0];
            // this row's query position and head (packed: the group's heads
            // share the tile, and its rows share one diagonal key tile)
            const int qpos = kPack ? mt * (128 / a.group) + row / a.group : mt * 128 + row;
            const int qh = kPack ? U.h * a.group + row % a.group : U.h;
            const int t0 = x ? U.t0[1] : U.t0[0];
            const int t1 = kExt ? (x ? U.t1[1] : U.t1[0]) : U.T;
            // this row's visible keys (rows past N: any non-empty range)
            int klo = 0, khi = a.N;
            if constexpr (kExt) {
                const int gr = min(mt * 128 + row, a.N - 1);
                klo = window_lo(gr, a);
                khi = window_hi(gr, a);
            }
            // FP8: the Q tile's scale and the largest V scale of the head
            // (the per-tile V scales are folded into P relative to it).
            // FP8 scales: Q per query head, K and V per K/V head (grouped heads)
            const size_t sbase = (static_cast<size_t>(U.b) * a.H + U.h) * a.n_kv;
            const size_t kvbase =
                kFP8 ? (static_cast<size_t>(U.b) * (a.H / a.group) + U.h / a.group) * a.n_kv : 0;
            float qs = 1.f, vmax = 1.f;
            if constexpr (kFP8) {
                qs = a.q_scale[sbase + mt];
                float vm = 0.f;
                for (int jj = lane; jj < a.n_kv; jj += 32) vm = fmaxf(vm, a.v_scale[kvbase + jj]);
#pragma unroll
                for (int m = 16; m > 0; m >>= 1) vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, m));
                vmax = vm;
            }
            // r: reference point (scaled log2 units); le: row sum of the FP32
            // exponentials (for LSE); lr: row sum of the same values rounded
            // as the P V product sees them (normalises O; 16-bit P only).
            float r = -INFINITY, le = 0.f, lr = 0.f;
            // FP8, per key tile: the score scale to log2 units with the q and
            // k tile scales ("FlashAttention-3 on Hopper", sec. 6.3), the
            // exponent offset c + log2(v_j / v_max) that carries the V tile
            // scale, and v_max / v_j for the row sum.  The next tile's scales
            // are loaded at the top of a tile (they land during the wait for
            // S) and turned into its constants after this tile's row sums:
            // neither the loads nor the division and logarithm sit on the
            // path from S to P'.
            float ks_n = 0.f, vs_n = 0.f;
            float sc_n = 0.f, voff_n = 0.f, ivr_n = 1.f;
            auto tile_load = [&](const int jj) __attribute__((always_inline)) {
                ks_n = a.k_scale[kvbase + jj];
                vs_n = a.v_scale[kvbase + jj];
            };
            auto tile_consts = [&]() __attribute__((always_inline)) {
                sc_n = sl2 * qs * ks_n;
                voff_n = C::P_OFFSET + log2f(vs_n / vmax);
                ivr_n = vmax / vs_n;
            };
            if (kFP8 && t0 < t1) {
                tile_load(U.jhi - 1 - t0);
                tile_consts();
            }
            for (int t = t0; t < t1; ++t) {
                const int j = U.jhi - 1 - t;
                const float sc_c = sc_n, voff_c = voff_n, ivr_c = ivr_n;
                if (kFP8 && t + 1 < t1) tile_load(j - 1);
                ok = mbar_wait(bar(C::B_SFULL + x), sph, w, 20);
                if (__any_sync(0xffffffffu, !ok)) { ok = false; break; }
                sph ^= 1;
                tc_fence_after();
                uint32_t s[128];
                float *sf = reinterpret_cast<float *>(s);
                // ---- S -> registers, masks: sequence tail and causal diagonal
                //      (variants: the row's window [klo, khi), after the
                //      softcap -- "FlashAttention-3 on Hopper", sec. 4.7:
                //      a score transformation precedes the mask) ----
                int lim = 128, llo = 0;
                if constexpr (kExt) {
                    lim = min(lim, khi - j * 128);
                    llo = klo - j * 128;
                } else {
                    if (j == a.n_kv - 1) lim = min(lim, a.N - j * 128);
                    if constexpr (kPack) {
                        if (kCausal && j == ((mt * (128 / a.group)) >> 7)) lim = min(lim, qpos - j * 128 + 1);
                    } else {
                        if (kCausal && j == mt) lim = min(lim, row + 1);
                    }
                }
                auto load_s = [&]() __attribute__((always_inline)) {
                    tmem_ld32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
                    tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
                    tmem_ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(&s[64]));
                    tmem_ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(&s[96]));
                    tmem_ld_wait();
                    if constexpr (kExt) {
                        if constexpr (kCap) {
#pragma unroll
                            for (int c = 0; c < 128; ++c) sf[c] = tanh_approx(sf[c] * sc_pre);
                        }
                        if (lim < 128 || llo > 0) {
#pragma unroll
                            for (int c = 0; c < 128; ++c)
                                if (c >= lim || c < llo) sf[c] = -INFINITY;
                        }
                    } else {
                        if (lim < 128) {
#pragma unroll
                            for (int c = 0; c < 128; ++c) if (c >= lim) sf[c] = -INFINITY;
                        }
                    }
                };
                load_s();
                auto row_max = [&]() __attribute__((always_inline)) -> float {
                    float m0 = sf[0], m1 = sf[1], m2 = sf[2], m3 = sf[3];
#pragma unroll
                    for (int c = 4; c < 128; c += 8) {
                        m0 = max3(m0, sf[c + 0], sf[c + 4]);
                        m1 = max3(m1, sf[c + 1], sf[c + 5]);
                        m2 = max3(m2, sf[c + 2], sf[c + 6]);
                        m3 = max3(m3, sf[c + 3], sf[c + 7]);
                    }
                    return fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
                };
                // r: reference of this tile's P; corr = 2^(r_old - r) rescales O
                // and the row sums when r moves.
                float rn = r, corr = 1.f;
                bool need = false;
                float2 e_a, e_b;
                uint32_t p[kFP8 ? 32 : 64];
                if constexpr (kFP8) {
                    const float sc = sc_c, voff = voff_c;
                    // e4m3 saturates above 448, so the row max comes first.
                    const float bnew = row_max() * sc;             // -inf stays -inf
                    if (r == -INFINITY) rn = bnew;
                    else { rn = (bnew > r + C::TAU) ? bnew : r; corr = ex2_approx(r - rn); }
                    need = (r != -INFINITY) && (rn != r);
                    const float rs = (rn == -INFINITY) ? 0.f : rn;
                    const float2 c2 = make_float2(sc, sc);
                    const float2 nr2 = make_float2(voff - rs, voff - rs);
                    e_a = make_float2(0.f, 0.f);
                    e_b = e_a;
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
                    tmem_st32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&p[0]));
                } else {
                    // ---- 16-bit P = 2^(x - r): first against the current r;
                    //      the max is formed only on the first tile or when
                    //      the tile's sum exceeds KEEP_SUM ----
                    const float2 c2 = make_float2(sl2, sl2);
                    auto exps = [&](const float rs) __attribute__((always_inline)) {
                        const float2 nr2 = make_float2(-rs, -rs);
                        e_a = make_float2(0.f, 0.f);
                        e_b = e_a;
#pragma unroll
                        for (int c = 0; c < 128; c += 4) {
                            const float2 x01 = __ffma2_rn(make_float2(sf[c + 0], sf[c + 1]), c2, nr2);
                            const float2 x23 = __ffma2_rn(make_float2(sf[c + 2], sf[c + 3]), c2, nr2);
                            const float2 e01 = make_float2(ex2_approx(x01.x), ex2_approx(x01.y));
                            const float2 e23 = make_float2(ex2_approx(x23.x), ex2_approx(x23.y));
                            p[c / 2] = pack2<kBF16>(e01.x, e01.y);
                            p[c / 2 + 1] = pack2<kBF16>(e23.x, e23.y);
                            e_a = __fadd2_rn(e_a, e01);
                            e_b = __fadd2_rn(e_b, e23);
                        }
                    };
                    bool keep = __all_sync(0xffffffffu, r != -INFINITY);
                    if (keep) {
                        exps(r);
                        const float ts = (e_a.x + e_a.y) + (e_b.x + e_b.y);
                        keep = __all_sync(0xffffffffu, ts <= C::KEEP_SUM);   // NaN: redo
                        if (!keep) load_s();
                    }
                    if (!keep) {
                        const float bnew = row_max() * sl2;
                        if (r == -INFINITY) rn = bnew;
                        else { rn = (bnew > r + C::TAU) ? bnew : r; corr = ex2_approx(r - rn); }
                        need = (r != -INFINITY) && (rn != r);
                        exps((rn == -INFINITY) ? 0.f : rn);
                    }
                    tmem_st32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&p[0]));
                    tmem_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&p[32]));
                }
                // ---- correction of O (its previous PV completed before S_FULL) ----
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
                    if constexpr (C::kLMMA) {            // L holds the rounded-P row sum
                        uint32_t lv[16];
                        tmem_ld16(tL, lv);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            lv[i] = __float_as_uint(__uint_as_float(lv[i]) * corr);
                        tmem_st16(tL, lv);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::B_PFULL + x));
                // ---- row sums, after P is published ----
                // (FP8: the row sum counts 2^(x - r + c) without the V factor)
                // (the row-sum updates are explicit fused multiply-adds: every
                // instantiation then rounds them alike, whatever the compiler
                // would contract)
                le = __fmaf_rn(le, corr, ((e_a.x + e_a.y) + (e_b.x + e_b.y)) * ivr_c);
                if constexpr (!kFP8 && !C::kLMMA) {
                    float2 r_a = make_float2(0.f, 0.f), r_b = r_a;
#pragma unroll
                    for (int i = 0; i < 64; i += 2) {
                        add_pair<kBF16>(r_a.x, r_a.y, p[i]);
                        add_pair<kBF16>(r_b.x, r_b.y, p[i + 1]);
                    }
                    lr = __fmaf_rn(lr, corr, (r_a.x + r_a.y) + (r_b.x + r_b.y));
                }
                r = rn;
                if (kFP8 && t + 1 < t1) tile_consts();
            }
            if (!ok) break;
            // ---- the row's normaliser and LSE ----
            // 16-bit P: O / l_r.  FP8: O v_max / l (O accumulated P' = P v_j/v_max).
            // (d = 64: l_r is the L accumulator, read with O below.)
            bool live = false;
            float inv = 0.f, lse2 = -INFINITY;      // LSE in log2 units
            auto normalise = [&]() __attribute__((always_inline)) {
                live = (le > 0.f) && (kFP8 || lr > 0.f);
                inv = live ? (kFP8 ? vmax / le : 1.f / lr) : 0.f;
                lse2 = live ? r - C::P_OFFSET + log2f(le) : -INFINITY;
                if constexpr (kExt) {
                    // Sink ("FlashAttention-3 on Hopper", sec. 4.6): one more
                    // term 2^(sigma log2 e - r) in both row sums, no value.
                    if (a.sinks != nullptr) {
                        const float sg = a.sinks[U.h] * 1.44269504088896340736f;
                        if (!live) {
                            inv = 0.f;
                            lse2 = sg;
                        } else {
                            const float M = fmaxf(r, sg);
                            lse2 = M + log2f(__fmaf_rn(le, ex2_approx(r - M), ex2_approx(sg - M)));
                            inv = 1.f / (lr + ex2_approx(sg - r));    // 2^+big -> inf -> 0
                        }
                    }
                }
            };
            if constexpr (!C::kLMMA) normalise();
            const int grow = qpos;
            {
                // ---- epilogue: O / l -> global ----
                ok = mbar_wait(bar(C::B_OFULL + x), oph, w, 21);
                if (__any_sync(0xffffffffu, !ok)) { ok = false; break; }
                oph ^= 1;
                tc_fence_after();
                // The whole O row comes into registers first, so the
                // accumulator is handed back to the next unit's P V before
                // the stores.
                uint32_t ov[D];
#pragma unroll
                for (int ch = 0; ch < D / 32; ++ch)
                    tmem_ld32(tO + ch * 32, *reinterpret_cast<uint32_t(*)[32]>(&ov[ch * 32]));
                if constexpr (C::kLMMA) {
                    uint32_t lv[16];
                    tmem_ld16(tL, lv);
                    tmem_ld_wait();
                    lr = __uint_as_float(lv[0]);
                    normalise();
                } else {
                    tmem_ld_wait();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::B_OEMPTY + x));
                if (grow < a.N) {
                    if constexpr (kSplit) {
                        // split key range: FP32 partial O
                        float *prow = a.o_part +
                            (((static_cast<size_t>(U.s) * a.B + U.b) * a.N + grow) * a.H + U.h) * D;
                        if (v8ok) {
#pragma unroll
                            for (int ch = 0; ch < D / 8; ++ch) {
                                uint32_t pv[8];
#pragma unroll
                                for (int i = 0; i < 8; ++i)
                                    pv[i] = __float_as_uint(__uint_as_float(ov[8 * ch + i]) * inv);
                                st_global_v8(prow + 8 * ch, pv);
                            }
                        } else {
#pragma unroll
                            for (int ch = 0; ch < D / 4; ++ch)
                                reinterpret_cast<float4 *>(prow)[ch] = make_float4(
                                    __uint_as_float(ov[4 * ch]) * inv, __uint_as_float(ov[4 * ch + 1]) * inv,
                                    __uint_as_float(ov[4 * ch + 2]) * inv,
                                    __uint_as_float(ov[4 * ch + 3]) * inv);
                        }
                    } else {
                        uint16_t *orow = reinterpret_cast<uint16_t *>(a.o) +
                                         ((static_cast<size_t>(U.b) * a.N + grow) * a.H + qh) * D;
                        if (v8ok) {
#pragma unroll
                            for (int ch = 0; ch < D / 16; ++ch) {
                                uint32_t pk[8];
#pragma unroll
                                for (int i = 0; i < 8; ++i)
                                    pk[i] = pack2<kBF16>(__uint_as_float(ov[16 * ch + 2 * i]) * inv,
                                                         __uint_as_float(ov[16 * ch + 2 * i + 1]) * inv);
                                st_global_v8(orow + 16 * ch, pk);
                            }
                        } else {
#pragma unroll
                            for (int ch = 0; ch < D / 8; ++ch) {
                                uint32_t pk[4];
#pragma unroll
                                for (int i = 0; i < 4; ++i)
                                    pk[i] = pack2<kBF16>(__uint_as_float(ov[8 * ch + 2 * i]) * inv,
                                                         __uint_as_float(ov[8 * ch + 2 * i + 1]) * inv);
                                reinterpret_cast<uint4 *>(orow)[ch] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                            }
                        }
                    }
                }
            }
            if constexpr (kSplit) {
                // split key range: the partial's LSE
                if (grow < a.N)
                    a.lse_part[((static_cast<size_t>(U.s) * a.B + U.b) * a.H + U.h) * a.N + grow] =
                        live ? (r + log2f(le)) * 0.69314718055994530942f : -INFINITY;
                continue;
            }
            if (a.lse != nullptr && grow < a.N)
                a.lse[(static_cast<size_t>(U.b) * a.H + qh) * a.N + grow] =
                    lse2 * 0.69314718055994530942f;
        }
    }

    // ---- teardown ----
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tbase, C::TMEM_COLS);
    }
}

}  // namespace fa
