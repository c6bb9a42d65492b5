// fa_device.cuh -- thin inline-PTX wrappers for sm_103a: mbarrier, TMA
// (cp.async.bulk.tensor), tcgen05 (alloc / mma / commit / ld / st / fences)
// and shared-memory matrix descriptors.  Every wait is bounded: it gives up
// after a wall-clock limit, records a status code in a device word and
// returns false, so no kernel can spin forever.
#pragma once

#include <cuda.h>
#include <cstdint>

namespace fa {

// ---------------------------------------------------------------------------
// Status word (owned by the host library; the kernel gets its address).
// ---------------------------------------------------------------------------
enum : uint32_t {
    kStatusOk = 0,
    kStatusTimeout = 1,
};

// Roles that may report a timeout (stored in status[1] for diagnosis).
enum : uint32_t {
    kRoleSoftmax0 = 1, kRoleSoftmax1 = 2, kRoleProducer = 3, kRoleMma = 4,
    kRoleDrain = 5, kRoleQuant = 6, kRoleSelftest = 7,
};

// A bounded wait gives up after this many nanoseconds of %globaltimer.
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count));
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];"
                 :: "r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 :: "r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// Shared per-CTA abort flag: once any role gives up, every other wait in the
// CTA returns false promptly instead of running into its own time limit.
struct WaitCtx {
    volatile uint32_t *abort_flag;   // in shared memory
    uint32_t *status;                // device status word (4 x u32)
    uint32_t role;
};

static __device__ __noinline__ void report_timeout(volatile uint32_t *abort_flag,
                                                   uint32_t *status, uint32_t role,
                                                   uint32_t where) {
    *abort_flag = 1u;
    if (atomicCAS(&status[0], kStatusOk, kStatusTimeout) == kStatusOk) {
        status[1] = role;
        status[2] = where;
        status[3] = blockIdx.x;
    }
    __threadfence();
}

// Waits until the phase of `bar` with parity `parity` has completed.
// Returns false (after recording a timeout) if it did not within the limit
// or if another role of this CTA has already given up.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          const WaitCtx &w, uint32_t where) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 31u) == 0u) {
            if (*w.abort_flag) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
                report_timeout(w.abort_flag, w.status, w.role, where);
                return false;
            }
        }
    }
}

// Whole-warp form of mbar_wait: every lane polls, the result is uniform.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity,
                                               const WaitCtx &w, uint32_t where) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, w, where));
}

// Bounded wait used only on the abort/teardown path: no reporting.
__device__ __forceinline__ bool mbar_wait_quiet(uint32_t bar, uint32_t parity,
                                                uint64_t limit_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
    return true;
}

// ---------------------------------------------------------------------------
// TMA (tensor maps are __grid_constant__ kernel parameters)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *m) {
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 4-D tiled load of box {c0.., c1.., c2.., c3..} into shared memory; the
// transaction bytes complete on `bar`.  c0 (innermost) must be 16-B aligned
// in bytes: every caller passes a multiple of 64 elements.
__device__ __forceinline__ void tma_load_4d(const CUtensorMap *m, uint32_t dst,
                                            uint32_t bar, int c0, int c1, int c2,
                                            int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2),
           "r"(c3), "r"(bar)
        : "memory");
}

// 32-byte store of eight 32-bit words (the address 32-byte aligned).
__device__ __forceinline__ void st_global_v8(void *p, const uint32_t *v) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                 :: "l"(p), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
                    "r"(v[6]), "r"(v[7])
                 : "memory");
}

// Cluster launch control (dynamic persistent scheduling): ask the hardware
// to cancel one not-yet-launched CTA of this grid; the 16-byte response
// lands in shared memory at resp and completes 16 transaction bytes on bar
// (armed by the caller with mbar_arrive_expect_tx).  A CTA that was
// cancelled never runs, so its block index becomes this CTA's work.
__device__ __forceinline__ void clc_try_cancel(uint32_t resp, uint32_t bar) {
    asm volatile(
        "clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128 "
        "[%0], [%1];" :: "r"(resp), "r"(bar) : "memory");
}
// The block index a completed response names, or -1 when nothing was
// cancelled (every CTA of the grid has been launched).
__device__ __forceinline__ int clc_block(uint32_t resp) {
    uint32_t ok, cx;
    asm volatile(
        "{\n\t.reg .b128 r;\n\t.reg .pred p;\n\t"
        "ld.shared.b128 r, [%2];\n\t"
        "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, r;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t"
        "clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %1, r;\n\t}"
        : "=r"(ok), "=r"(cx) : "r"(resp) : "memory");
    return ok ? static_cast<int>(cx) : -1;
}

// The dynamic causal order (clc_try_cancel schedules it): groups of chunk
// heads, longest unit first within a group, every head's shortest unit last.
// Position u over BH heads of n units each (unit i of a head is its
// (i+1)-th shortest): the unit index i and the head bh.
__device__ __forceinline__ void dynamic_order(int u, int BH, int n, int chunk, int &i, int &bh) {
    const int n1 = n - 1;                          // units per head before the tail
    const int grouped = BH * n1;
    if (u < grouped) {
        const int g = u / (chunk * n1);
        const int r = u - g * chunk * n1;
        const int cg = min(chunk, BH - g * chunk); // heads in this group
        i = n1 - r / cg;
        bh = g * chunk + r % cg;
    } else {
        i = 0;
        bh = u - grouped;
    }
}

// 4-D tiled store of a box from shared memory (bulk-group completion).  Out-of-
// range parts of the box are not written; every coordinate is >= 0 and c0
// is 16-byte aligned in bytes.
__device__ __forceinline__ void tma_store_4d(const CUtensorMap *m, uint32_t src, int c0,
                                             int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%1, %2, %3, %4}], [%5];"
        :: "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(src)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until the committed bulk stores have read their shared-memory source.
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Waits until the committed bulk stores have completed.
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) reads of them.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05
// ---------------------------------------------------------------------------
// Whole-warp TMEM allocation; the base address is written to `dst_smem`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(dst_smem), "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                 :: "r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]; kind::f16 (bf16/fp16 in, fp32 acc)
__device__ __forceinline__ void mma_ss_f16(uint32_t d_tmem, uint64_t a_desc,
                                           uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]; kind::f16
__device__ __forceinline__ void mma_ts_f16(uint32_t d_tmem, uint32_t a_tmem,
                                           uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Warp-converged forms: the whole warp executes the statement and the
// lane chosen by elect.sync (the lowest lane of a full warp, so always the
// same lane) issues it.  Keeping the issuing warp converged lets descriptor
// arithmetic stay warp-uniform; one divergent lane issuing tcgen05.mma was
// measured at ~54 cycles per instruction versus ~21 for this form, against
// 64 cycles of tensor work for a 128x128x16 MMA.
__device__ __forceinline__ void mma_ss_f16_elect(uint32_t d_tmem, uint64_t a_desc,
                                                 uint64_t b_desc, uint32_t idesc,
                                                 uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred e, p;\n\telect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_ts_f16_elect(uint32_t d_tmem, uint32_t a_tmem,
                                                 uint64_t b_desc, uint32_t idesc,
                                                 uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred e, p;\n\telect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// kind::f8f6f4 forms (e4m3 x e4m3 -> f32), same issue discipline.
__device__ __forceinline__ void mma_ss_f8_elect(uint32_t d_tmem, uint64_t a_desc,
                                                uint64_t b_desc, uint32_t idesc,
                                                uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred e, p;\n\telect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_ts_f8_elect(uint32_t d_tmem, uint32_t a_tmem,
                                                uint64_t b_desc, uint32_t idesc,
                                                uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred e, p;\n\telect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}"
        :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit_elect(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}"
        :: "r"(bar) : "memory");
}

// Arrive (once) on `bar` when every tcgen05 MMA issued so far by this thread
// has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
        :: "r"(bar) : "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (the layout TMA writes
// with CU_TENSOR_MAP_SWIZZLE_128B into a 1024-B aligned buffer).
//   bits  0-13 start address >> 4      bits 16-29 leading byte offset >> 4
//   bits 32-45 stride byte offset >> 4 bits 46-47 descriptor version (1)
//   bits 49-51 base offset (0)         bit  52    LBO mode (0)
//   bits 61-63 layout (2 = 128-B swizzle)
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                    uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor for kind::f16 with FP32 accumulation.
//   bits 4-5 D format (1 = f32), 7-9 A format, 10-12 B format
//   (0 = f16, 1 = bf16), bit 15 A major, bit 16 B major (0 = K, 1 = MN),
//   bits 17-22 N >> 3, bits 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_f16(uint32_t M, uint32_t N, bool bf16,
                                                 bool a_mn_major, bool b_mn_major) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
           ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
           ((N >> 3) << 17) | ((M >> 4) << 24);
}

// Instruction descriptor for kind::f8f6f4, e4m3 x e4m3 -> f32.
__host__ __device__ constexpr uint32_t idesc_e4m3(uint32_t M, uint32_t N,
                                                  bool a_mn_major, bool b_mn_major) {
    return (1u << 4) | (0u << 7) | (0u << 10) |
           ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
           ((N >> 3) << 17) | ((M >> 4) << 24);
}

// TMEM loads/stores, 32 lanes x 32 bits shape: thread t of the warp accesses
// lane (addr.lane + t); .xN covers N consecutive 32-bit columns.
#define FA_R8(a, i) "=r"(a[i + 0]), "=r"(a[i + 1]), "=r"(a[i + 2]), "=r"(a[i + 3]), \
                    "=r"(a[i + 4]), "=r"(a[i + 5]), "=r"(a[i + 6]), "=r"(a[i + 7])
#define FA_W8(a, i) "r"(a[i + 0]), "r"(a[i + 1]), "r"(a[i + 2]), "r"(a[i + 3]), \
                    "r"(a[i + 4]), "r"(a[i + 5]), "r"(a[i + 6]), "r"(a[i + 7])

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : FA_R8(r, 0), FA_R8(r, 8), FA_R8(r, 16), FA_R8(r, 24)
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
        :: "r"(taddr), FA_W8(r, 0), FA_W8(r, 8), FA_W8(r, 16), FA_W8(r, 24)
        : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : FA_R8(r, 0), FA_R8(r, 8)
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t *r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        :: "r"(taddr), FA_W8(r, 0), FA_W8(r, 8)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

#undef FA_R8
#undef FA_W8

// ---------------------------------------------------------------------------
// Register reallocation between warpgroups (all four warps of a warpgroup
// execute the same instruction).  The sum over warpgroups must not exceed the
// registers the block was launched with.
// ---------------------------------------------------------------------------
template <uint32_t N>
__device__ __forceinline__ void regs_grow() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" :: "n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_shrink() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" :: "n"(N));
}

// ---------------------------------------------------------------------------
// Arithmetic helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Hardware tanh (MUFU); its error bound is measured and stated where the
// softcap uses it.
__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Two FP32 values -> packed pair of 16-bit floats (low half = a), RN.
template <bool kBF16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
    uint32_t r;
    if constexpr (kBF16) {
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    } else {
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    }
    return r;
}

// acc += lo + hi of a packed pair of 16-bit floats, each widened exactly,
// with mixed-precision adds (no separate unpacking).
template <bool kBF16>
__device__ __forceinline__ void add_pair(float &acc0, float &acc1, uint32_t pk) {
    if constexpr (kBF16) {
        asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
            "add.rn.f32.bf16 %0, lo, %0;\n\tadd.rn.f32.bf16 %1, hi, %1;\n\t}"
            : "+f"(acc0), "+f"(acc1) : "r"(pk));
    } else {
        asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
            "add.rn.f32.f16 %0, lo, %0;\n\tadd.rn.f32.f16 %1, hi, %1;\n\t}"
            : "+f"(acc0), "+f"(acc1) : "r"(pk));
    }
}

// Four FP32 values -> four e4m3 bytes (RN, saturating at +-448), a first.
__device__ __forceinline__ uint32_t pack4_e4m3(float a, float b, float c, float d) {
    uint16_t lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// Inverse of pack2: the two 16-bit floats of a packed pair, widened exactly.
template <bool kBF16>
__device__ __forceinline__ void unpack2(uint32_t pk, float &lo, float &hi) {
    if constexpr (kBF16) {
        lo = __uint_as_float(pk << 16);
        hi = __uint_as_float(pk & 0xffff0000u);
    } else {
        asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
            "cvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
            : "=f"(lo), "=f"(hi) : "r"(pk));
    }
}

// Persistent unit order: CTA c of G runs units c, then c + s0, then
// c + s0 + (2G - s0), ... -- strides that alternate between s0 and 2G - s0.
// Plain orders take s0 = G (units c, c + G, c + 2G, ...).  Longest-first
// orders go back and forth over the CTAs, s0 = 2G - 1 - 2c: round k gives
// CTA c unit kG + c for even k and kG + G - 1 - c for odd k, so a CTA that
// takes one of the longest units of a round takes one of the shortest of
// the next (striding one way gave CTA 0 the longest unit of every round).
// The units a CTA visits only grow, so the first one past the end ends its
// sequence.  Every role of a CTA walks the same sequence:
//   for (int u = blockIdx.x, st = unit_stride0(snake); u < n;
//        u += st, st = 2 * gridDim.x - st)
__device__ __forceinline__ int unit_stride0(bool snake) {
    const int G = gridDim.x, c = blockIdx.x;
    return snake ? 2 * G - 1 - 2 * c : G;
}

}  // namespace fa
