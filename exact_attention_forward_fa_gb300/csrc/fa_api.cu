// fa_api.cu -- the C ABI declared in include/fa.h: argument validation,
// per-device properties, TMA tensor-map encoding, kernel selection, launch,
// and the device status word read by fa_check_status.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "fa.h"
#include "fa_launch.cuh"

namespace {

constexpr int kVersion = 100;   // 0.1.0

// Set by kernels whose bounded waits give up: [0] code, [1] role,
// [2] wait site, [3] block index.  One instance per device context.
__device__ uint32_t g_fa_status[4];

struct DeviceInfo {
    bool ready = false;
    int sm_count = 0;
    int cc_major = 0, cc_minor = 0;
    uint32_t *status = nullptr;   // device address of g_fa_status
};

constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;
uint32_t g_last_detail[4] = {0, 0, 0, 0};

// The workspace of fa_bwd_noalloc: a file-scope device array in the
// library's image, for callers that must not allocate device memory at the
// point of the call (a program whose device memory is reserved up front, a
// runtime that forbids allocation once a step has started).  Every device
// that loads the library holds its own copy until the process exits.  It
// bounds the problem: 2 * B * H * ceil(N/128) * 128 floats (D and LSE*log2 e,
// padded to whole tiles) must fit in 4 Mi floats (16 MiB).  Every element
// the backward reads is first written by its preprocess in the same call,
// so nothing needs to start at zero.  All calls on a device share the
// array: calls that overlap in time (other streams, other host threads)
// race on it.  Its device address is resolved once per device, on the first
// call with that device current, and cached; after a cudaDeviceReset the
// cached address is stale, so the entry point must not be used after one in
// the same process.
constexpr size_t kNoallocWorkspaceFloats = size_t(1) << 22;
static __device__ __align__(256) float g_noalloc_workspace[kNoallocWorkspaceFloats];
float *g_noalloc_ptr[kMaxDevices] = {};

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

fa_status get_device(DeviceInfo **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo &d = g_dev[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return FA_ERR_CUDA;
        void *sym = nullptr;
        if (cudaGetSymbolAddress(&sym, g_fa_status) != cudaSuccess) return FA_ERR_CUDA;
        d.status = static_cast<uint32_t *>(sym);
        if (g_encode == nullptr) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q) != cudaSuccess ||
                q != cudaDriverEntryPointSuccess || fn == nullptr)
                return FA_ERR_CUDA;
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
        d.ready = true;
    }
    if (!(d.cc_major == 10 && d.cc_minor == 3)) return FA_ERR_UNSUPPORTED;
    *out = &d;
    return FA_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 4-D map over a [B][N][H][d] tensor: dims {d, H, N, B}, box {128 B of the
// row, 1, rows, 1}, 128-byte swizzle, rows beyond N read as zero.  2-byte
// elements (bf16/fp16) or 1-byte e4m3 codes.
fa_status encode_bshd(CUtensorMap *m, const void *ptr, CUtensorMapDataType dt, int B,
                      int H, int N, int d, cuuint32_t rows) {
    const cuuint64_t esz = dt == CU_TENSOR_MAP_DATA_TYPE_UINT8 ? 1 : 2;
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                          static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(B)};
    cuuint64_t strides[3] = {esz * d, esz * d * H, esz * d * H * static_cast<cuuint64_t>(N)};
    cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / esz), 1, rows, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = g_encode(m, dt, 4, const_cast<void *>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// The same map with the box {128 B, g heads, 128 / g rows, 1}: one box is
// a Q tile of g heads packed row by row (tile row p = position p / g,
// head p % g), 128 rows of 128 B in shared memory like an ordinary tile.
fa_status encode_bshd_packed(CUtensorMap *m, const void *ptr, CUtensorMapDataType dt, int B,
                             int H, int N, int d, int g) {
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                          static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(B)};
    cuuint64_t strides[3] = {2ull * d, 2ull * d * H, 2ull * d * H * static_cast<cuuint64_t>(N)};
    cuuint32_t box[4] = {64, static_cast<cuuint32_t>(g), static_cast<cuuint32_t>(128 / g), 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = g_encode(m, dt, 4, const_cast<void *>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

extern "C" {

int fa_version(void) { return kVersion; }

const char *fa_status_string(fa_status s) {
    switch (s) {
        case FA_OK: return "FA_OK";
        case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
        case FA_ERR_MISALIGNED: return "FA_ERR_MISALIGNED";
        case FA_ERR_TOO_LARGE: return "FA_ERR_TOO_LARGE";
        case FA_ERR_CUDA: return "FA_ERR_CUDA";
        case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
    }
    return "FA_ERR_UNKNOWN";
}

// The forward for H query heads over H_kv key/value heads (H_kv divides H;
// query head h reads key/value head h / (H / H_kv)).  pack: the g = H / H_kv
// query heads of a key/value head share each Q tile (d in {64, 128}, g
// dividing 128); with g = 1 that is the plain layout.
// Causal units (unsplit, unpacked; every head dim) run in the kernels'
// dynamic order: one CTA per unit (CTAs that have not started yet are taken
// over by running ones), and a.chunk query heads per group of the order, as
// many as keep the group's K and V within 32 MiB of L2.
static void set_dynamic_order(fa::FwdLaunch &L, uint64_t units, int B, int H, int N, int d,
                              int elem_bytes, int group) {
    L.grid = static_cast<int>(units);
    const uint64_t kv_head = 2ull * static_cast<uint64_t>(N) * d * elem_bytes;
    uint64_t c = (32ull << 20) / (kv_head > 0 ? kv_head : 1) * static_cast<uint64_t>(group);
    const uint64_t bh = static_cast<uint64_t>(B) * H;
    if (c < 1) c = 1;
    if (c > bh) c = bh;
    L.args.chunk = static_cast<int>(c);
}

static fa_status fwd_impl(const void *q, const void *k, const void *v, void *o, float *lse,
                          int B, int H, int H_kv, int N, int d, float alpha, int causal,
                          fa_dtype dtype, void *stream, bool pack = false) {
    // ---- host-side validation: nothing is launched on failure ----
    if (!q || !k || !v || !o) return FA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || N < 1 || d < 1) return FA_ERR_INVALID_ARG;
    if (H_kv < 1 || H % H_kv != 0) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(alpha)) return FA_ERR_INVALID_ARG;
    if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FA_ERR_MISALIGNED;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return FA_ERR_MISALIGNED;
    const int g = H / H_kv;
    if (pack && g == 1) pack = false;                  // one head per tile: the plain layout
    if (pack && (d == 256 || 128 % g != 0)) return FA_ERR_UNSUPPORTED;
    // TMA: every global stride < 2^40 bytes; kernel indexing uses 64-bit
    // offsets, the unit counter is a 32-bit int.
    const uint64_t batch_stride = 2ull * d * H * static_cast<uint64_t>(N);
    if (batch_stride >= (1ull << 40)) return FA_ERR_TOO_LARGE;
    // Work units: pairs of 128-row Q tiles for d <= 128, single Q tiles
    // for d = 256 (whose O accumulator alone fills half of TMEM); packed,
    // pairs of tiles of 128 / g positions over the key/value heads.
    const uint64_t n_qt = (static_cast<uint64_t>(N) + 127) / 128;
    const uint64_t n_pt = pack ? (static_cast<uint64_t>(N) + 128 / g - 1) / (128 / g) : n_qt;
    const uint64_t units = pack ? static_cast<uint64_t>(B) * H_kv * ((n_pt + 1) / 2)
                                : static_cast<uint64_t>(B) * H * (d == 256 ? n_qt : (n_qt + 1) / 2);
    if (units > 0x7fffffffull || static_cast<uint64_t>(B) * H * N > 0x7fffffffffffull)
        return FA_ERR_TOO_LARGE;

    DeviceInfo *dev = nullptr;
    fa_status st = get_device(&dev);
    if (st != FA_OK) return st;

    fa::FwdLaunch L;
    std::memset(&L, 0, sizeof(L));
    const CUtensorMapDataType dt =
        dtype == FA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const cuuint32_t kv_rows = d == 256 ? 64 : 128;     // key tile height
    st = pack ? encode_bshd_packed(&L.q, q, dt, B, H, N, d, g) : encode_bshd(&L.q, q, dt, B, H, N, d, 128);
    if (st != FA_OK) return st;
    if ((st = encode_bshd(&L.k, k, dt, B, H_kv, N, d, kv_rows)) != FA_OK) return st;
    if ((st = encode_bshd(&L.v, v, dt, B, H_kv, N, d, kv_rows)) != FA_OK) return st;
    L.args.o = o;
    L.args.lse = lse;
    L.args.status = dev->status;
    L.args.B = B;
    L.args.H = H;
    L.args.N = N;
    L.args.n_kv = static_cast<int>(d == 256 ? (static_cast<uint64_t>(N) + 63) / 64 : n_qt);
    L.args.n_pairs = static_cast<int>((n_pt + 1) / 2);
    L.args.n_units = static_cast<int>(units);
    L.args.group = H / H_kv;
    L.args.n_splits = 1;
    L.args.scale_log2 = static_cast<float>(static_cast<double>(alpha) * 1.4426950408889634);
    L.grid = static_cast<int>(units < static_cast<uint64_t>(dev->sm_count) ? units : dev->sm_count);
    L.args.chunk = 1;
    if (causal && !pack) set_dynamic_order(L, units, B, H, N, d, 2, g);
    L.stream = static_cast<cudaStream_t>(stream);
    L.causal = causal != 0;
    L.bf16 = dtype == FA_BF16;
    L.d64 = d == 64;

    cudaError_t e = pack ? fa::launch_fwd_pack(L)
                    : (d == 64) ? fa::launch_fwd_d64(L)
                    : (d == 128) ? fa::launch_fwd_d128(L) : fa::launch_fwd_d256(L);
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                 int H, int N, int d, float alpha, int causal, fa_dtype dtype,
                 void *stream) {
    return fwd_impl(q, k, v, o, lse, B, H, H, N, d, alpha, causal, dtype, stream);
}

fa_status fa_fwd_gqa_packed(const void *q, const void *k, const void *v, void *o, float *lse,
                            int B, int H, int H_kv, int N, int d, float alpha, int causal,
                            fa_dtype dtype, void *stream) {
    return fwd_impl(q, k, v, o, lse, B, H, H_kv, N, d, alpha, causal, dtype, stream, true);
}

fa_status fa_fwd_gqa(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                     int H, int H_kv, int N, int d, float alpha, int causal, fa_dtype dtype,
                     void *stream) {
    return fwd_impl(q, k, v, o, lse, B, H, H_kv, N, d, alpha, causal, dtype, stream);
}

fa_status fa_fwd_ext(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                     int H, int H_kv, int N, int d, float alpha, int window_left,
                     int window_right, float softcap, const float *sinks, fa_dtype dtype,
                     void *stream) {
    // ---- host-side validation: nothing is launched on failure ----
    if (!q || !k || !v || !o) return FA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || N < 1 || d < 1) return FA_ERR_INVALID_ARG;
    if (H_kv < 1 || H % H_kv != 0) return FA_ERR_INVALID_ARG;
    if (window_left < -1 || window_right < -1) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(alpha) || !std::isfinite(softcap) || softcap < 0.f)
        return FA_ERR_INVALID_ARG;
    if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FA_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(sinks) & 3u))
        return FA_ERR_MISALIGNED;
    const uint64_t batch_stride = 2ull * d * H * static_cast<uint64_t>(N);
    if (batch_stride >= (1ull << 40)) return FA_ERR_TOO_LARGE;
    const uint64_t n_qt = (static_cast<uint64_t>(N) + 127) / 128;
    const uint64_t units = static_cast<uint64_t>(B) * H * ((n_qt + 1) / 2);
    if (units > 0x7fffffffull || static_cast<uint64_t>(B) * H * N > 0x7fffffffffffull)
        return FA_ERR_TOO_LARGE;
    // alpha / c must stay a finite float for the softcap's first constant
    const double pre = softcap > 0.f ? static_cast<double>(alpha) / softcap : 0.0;
    if (!std::isfinite(static_cast<float>(pre))) return FA_ERR_INVALID_ARG;

    DeviceInfo *dev = nullptr;
    fa_status st = get_device(&dev);
    if (st != FA_OK) return st;

    fa::FwdLaunch L;
    std::memset(&L, 0, sizeof(L));
    const CUtensorMapDataType dt =
        dtype == FA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    if ((st = encode_bshd(&L.q, q, dt, B, H, N, d, 128)) != FA_OK) return st;
    if ((st = encode_bshd(&L.k, k, dt, B, H_kv, N, d, 128)) != FA_OK) return st;
    if ((st = encode_bshd(&L.v, v, dt, B, H_kv, N, d, 128)) != FA_OK) return st;
    L.args.o = o;
    L.args.lse = lse;
    L.args.status = dev->status;
    L.args.B = B;
    L.args.H = H;
    L.args.N = N;
    L.args.n_kv = static_cast<int>(n_qt);
    L.args.n_pairs = static_cast<int>((n_qt + 1) / 2);
    L.args.n_units = static_cast<int>(units);
    L.args.group = H / H_kv;
    L.args.n_splits = 1;
    L.args.scale_log2 = static_cast<float>(static_cast<double>(alpha) * 1.4426950408889634);
    L.args.wl = window_left;
    L.args.wr = window_right;
    L.args.sc_pre = static_cast<float>(pre);
    L.args.sc_post = static_cast<float>(static_cast<double>(softcap) * 1.4426950408889634);
    L.args.sinks = sinks;
    L.grid = static_cast<int>(units < static_cast<uint64_t>(dev->sm_count) ? units : dev->sm_count);
    L.stream = static_cast<cudaStream_t>(stream);
    L.bf16 = dtype == FA_BF16;
    L.d64 = d == 64;
    cudaError_t e = softcap > 0.f ? fa::launch_fwd_ext_softcap(L) : fa::launch_fwd_ext(L);
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// Split-KV: workspace floats for S splits (partial O in FP32 plus LSE).
static uint64_t splitkv_floats(uint64_t B, uint64_t H, uint64_t N, uint64_t d, uint64_t S) {
    return S * B * N * H * d + S * B * H * N;
}

long long fa_splitkv_workspace_floats(int B, int H, int N, int d, int n_splits) {
    if (B < 1 || H < 1 || N < 1 || d < 1 || n_splits < 1) return -1;
    return static_cast<long long>(splitkv_floats(B, H, N, d, n_splits));
}

int fa_splitkv_auto(int B, int H, int N, int d) {
    if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128)) return 1;
    DeviceInfo *dev = nullptr;
    if (get_device(&dev) != FA_OK) return 1;
    const long long n_kv = (N + 127) / 128;
    const long long units = static_cast<long long>(B) * H * ((n_kv + 1) / 2);
    const long long sm = dev->sm_count;
    // Measured on GB300: splitting pays only while every split unit still
    // runs in one wave -- a second wave repeats each unit's fixed cost.  So:
    // the fewest splits that occupy >= 80 % of the SMs, at most one wave,
    // at least 4 key tiles per split, at most 16.
    if (units * 5 >= sm * 4) return 1;
    long long s = (sm * 4 + units * 5 - 1) / (units * 5);
    s = s < sm / units ? s : sm / units;
    s = s < n_kv / 4 ? s : n_kv / 4;
    s = s < 16 ? s : 16;
    return static_cast<int>(s < 1 ? 1 : s);
}

fa_status fa_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse,
                         int B, int H, int N, int d, float alpha, int causal, fa_dtype dtype,
                         int n_splits, float *workspace, void *stream) {
    // ---- host-side validation: nothing is launched on failure ----
    if (!q || !k || !v || !o || !workspace) return FA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || N < 1 || d < 1) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(alpha)) return FA_ERR_INVALID_ARG;
    if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_INVALID_ARG;
    if (n_splits < 1 || n_splits > 16) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(workspace))
        return FA_ERR_MISALIGNED;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return FA_ERR_MISALIGNED;
    const uint64_t batch_stride = 2ull * d * H * static_cast<uint64_t>(N);
    if (batch_stride >= (1ull << 40)) return FA_ERR_TOO_LARGE;
    const uint64_t n_qt = (static_cast<uint64_t>(N) + 127) / 128;
    const uint64_t units = static_cast<uint64_t>(n_splits) * B * H * ((n_qt + 1) / 2);
    if (units > 0x7fffffffull ||
        splitkv_floats(B, H, N, d, n_splits) > 0x3fffffffffffull)
        return FA_ERR_TOO_LARGE;

    DeviceInfo *dev = nullptr;
    fa_status st = get_device(&dev);
    if (st != FA_OK) return st;

    fa::FwdLaunch L;
    std::memset(&L, 0, sizeof(L));
    const CUtensorMapDataType dt =
        dtype == FA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    if ((st = encode_bshd(&L.q, q, dt, B, H, N, d, 128)) != FA_OK) return st;
    if ((st = encode_bshd(&L.k, k, dt, B, H, N, d, 128)) != FA_OK) return st;
    if ((st = encode_bshd(&L.v, v, dt, B, H, N, d, 128)) != FA_OK) return st;
    float *o_part = workspace;
    float *lse_part = workspace + static_cast<size_t>(n_splits) * B * N * H * d;
    L.args.o = o;
    L.args.lse = nullptr;
    L.args.status = dev->status;
    L.args.B = B;
    L.args.H = H;
    L.args.N = N;
    L.args.n_kv = static_cast<int>(n_qt);
    L.args.n_pairs = static_cast<int>((n_qt + 1) / 2);
    L.args.n_units = static_cast<int>(units);
    L.args.group = 1;
    L.args.n_splits = n_splits;
    L.args.o_part = o_part;
    L.args.lse_part = lse_part;
    L.args.scale_log2 = static_cast<float>(static_cast<double>(alpha) * 1.4426950408889634);
    L.grid = static_cast<int>(units < static_cast<uint64_t>(dev->sm_count) ? units : dev->sm_count);
    L.stream = static_cast<cudaStream_t>(stream);
    L.causal = causal != 0;
    L.bf16 = dtype == FA_BF16;
    L.d64 = d == 64;
    cudaError_t e = fa::launch_fwd_split(L);
    if (e != cudaSuccess) return FA_ERR_CUDA;

    fa::CombineArgs c;
    c.o_part = o_part;
    c.lse_part = lse_part;
    c.o = o;
    c.lse = lse;
    c.B = B;
    c.H = H;
    c.N = N;
    c.d = d;
    c.S = n_splits;
    c.n_kv = static_cast<int>(n_qt);
    c.causal = causal;
    c.bf16 = dtype == FA_BF16;
    const uint64_t rows = static_cast<uint64_t>(B) * N * H;
    const uint64_t g = (rows + 7) / 8;                 // 8 rows (warps) per CTA
    const uint64_t gcap = 16ull * dev->sm_count;
    e = fa::launch_combine(c, static_cast<int>(g < gcap ? g : gcap), L.stream);
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

static fa_status quantize_impl(const void *x, uint8_t *x8, float *scales,
                               const float *hadamard_signs, int B, int H, int N, int d,
                               int granularity, void *stream) {
    if (!x || !x8 || !scales) return FA_ERR_INVALID_ARG;
    if (granularity < FA_SCALE_TILE || granularity > FA_SCALE_TENSOR) return FA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || N < 1 || d < 1) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(x8)) return FA_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(scales) & 3u) ||
        (reinterpret_cast<uintptr_t>(hadamard_signs) & 3u))
        return FA_ERR_MISALIGNED;
    const uint64_t n_tiles = (static_cast<uint64_t>(N) + 127) / 128;
    if (static_cast<uint64_t>(B) * H * n_tiles > 0x7fffffffull ||
        static_cast<uint64_t>(B) * H * N > 0x7fffffffffffull)
        return FA_ERR_TOO_LARGE;
    DeviceInfo *dev = nullptr;
    fa_status st = get_device(&dev);
    if (st != FA_OK) return st;
    fa::QuantLaunch L;
    std::memset(&L, 0, sizeof(L));
    // Without rotation one TMA box is a whole 128-row tile, {d, 1, 128, 1},
    // no swizzle.  With it, 128-byte column chunks {64, 1, 128, 1} in the
    // 128-byte swizzle (rows read by one thread each without conflicts), and
    // the codes leave through TMA stores of {128, 1, 128, 1} (64-byte swizzle
    // and {64, 1, 128, 1} at d = 64).
    if (hadamard_signs) {
        if ((st = encode_bshd(&L.x, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, B, H, N, d, 128)) != FA_OK)
            return st;
        const cuuint32_t w8 = d == 64 ? 64 : 128;
        cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(B)};
        cuuint64_t strides[3] = {1ull * d, 1ull * d * H, 1ull * d * H * static_cast<cuuint64_t>(N)};
        cuuint32_t box[4] = {w8, 1, 128, 1};
        cuuint32_t estr[4] = {1, 1, 1, 1};
        if (g_encode(&L.x8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, x8, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE,
                     d == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return FA_ERR_CUDA;
    } else {
        cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(B)};
        cuuint64_t strides[3] = {2ull * d, 2ull * d * H, 2ull * d * H * static_cast<cuuint64_t>(N)};
        cuuint32_t box[4] = {static_cast<cuuint32_t>(d), 1, 128, 1};
        cuuint32_t estr[4] = {1, 1, 1, 1};
        if (g_encode(&L.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(x), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return FA_ERR_CUDA;
    }
    L.args.x8 = x8;
    L.args.scales = scales;
    L.args.signs = hadamard_signs;
    L.args.status = dev->status;
    L.args.B = B;
    L.args.H = H;
    L.args.N = N;
    L.args.n_tiles = static_cast<int>(n_tiles);
    L.args.total = static_cast<int>(static_cast<uint64_t>(B) * H * n_tiles);
    L.d = d;
    L.sm_count = dev->sm_count;
    L.granularity = granularity;
    L.stream = static_cast<cudaStream_t>(stream);
    cudaError_t e = fa::launch_quantize(L);
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_quantize_fp8(const void *x, uint8_t *x8, float *scales,
                          const float *hadamard_signs, int B, int H, int N, int d,
                          void *stream) {
    return quantize_impl(x, x8, scales, hadamard_signs, B, H, N, d, FA_SCALE_TILE, stream);
}

fa_status fa_quantize_fp8_granular(const void *x, uint8_t *x8, float *scales,
                                   const float *hadamard_signs, int B, int H, int N, int d,
                                   int granularity, void *stream) {
    return quantize_impl(x, x8, scales, hadamard_signs, B, H, N, d, granularity, stream);
}

static fa_status fwd_fp8_impl(const uint8_t *q8, const uint8_t *k8, const uint8_t *v8,
                              const float *q_scale, const float *k_scale, const float *v_scale,
                              void *o, float *lse, int B, int H, int H_kv, int N, int d,
                              float alpha, int causal, void *stream) {
    if (!q8 || !k8 || !v8 || !q_scale || !k_scale || !v_scale || !o) return FA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || N < 1 || d < 1) return FA_ERR_INVALID_ARG;
    if (H_kv < 1 || H % H_kv != 0) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(alpha)) return FA_ERR_INVALID_ARG;
    if (d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
    if (!aligned16(q8) || !aligned16(k8) || !aligned16(v8) || !aligned16(o)) return FA_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(q_scale) & 3u) || (reinterpret_cast<uintptr_t>(k_scale) & 3u) ||
        (reinterpret_cast<uintptr_t>(v_scale) & 3u) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
        return FA_ERR_MISALIGNED;
    const uint64_t batch_stride = 1ull * d * H * static_cast<uint64_t>(N);
    if (batch_stride >= (1ull << 40)) return FA_ERR_TOO_LARGE;
    // work units: pairs of 128-row Q tiles at d = 128, single Q tiles at
    // d = 256 (whose O accumulator alone fills half of TMEM)
    const uint64_t n_qt = (static_cast<uint64_t>(N) + 127) / 128;
    const uint64_t units = static_cast<uint64_t>(B) * H * (d == 256 ? n_qt : (n_qt + 1) / 2);
    if (units > 0x7fffffffull || static_cast<uint64_t>(B) * H * N > 0x7fffffffffffull)
        return FA_ERR_TOO_LARGE;
    DeviceInfo *dev = nullptr;
    fa_status st = get_device(&dev);
    if (st != FA_OK) return st;

    fa::FwdLaunch L;
    std::memset(&L, 0, sizeof(L));
    const CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    if ((st = encode_bshd(&L.q, q8, dt, B, H, N, d, 128)) != FA_OK) return st;
    if ((st = encode_bshd(&L.k, k8, dt, B, H_kv, N, d, 128)) != FA_OK) return st;
    if ((st = encode_bshd(&L.v, v8, dt, B, H_kv, N, d, 128)) != FA_OK) return st;
    L.args.o = o;
    L.args.lse = lse;
    L.args.status = dev->status;
    L.args.B = B;
    L.args.H = H;
    L.args.N = N;
    L.args.n_kv = static_cast<int>(n_qt);
    L.args.n_pairs = static_cast<int>((n_qt + 1) / 2);
    L.args.n_units = static_cast<int>(units);
    L.args.group = H / H_kv;
    L.args.n_splits = 1;
    L.args.scale_log2 = static_cast<float>(static_cast<double>(alpha) * 1.4426950408889634);
    L.args.q_scale = q_scale;
    L.args.k_scale = k_scale;
    L.args.v_scale = v_scale;
    L.grid = static_cast<int>(units < static_cast<uint64_t>(dev->sm_count) ? units : dev->sm_count);
    L.args.chunk = 1;
    if (causal) set_dynamic_order(L, units, B, H, N, d, 1, H / H_kv);
    L.stream = static_cast<cudaStream_t>(stream);
    L.causal = causal != 0;
    L.bf16 = true;
    cudaError_t e = d == 256 ? fa::launch_fwd_fp8_d256(L) : fa::launch_fwd_fp8(L);
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_fwd_fp8(const uint8_t *q8, const uint8_t *k8, const uint8_t *v8,
                     const float *q_scale, const float *k_scale, const float *v_scale,
                     void *o, float *lse, int B, int H, int N, int d, float alpha,
                     int causal, void *stream) {
    return fwd_fp8_impl(q8, k8, v8, q_scale, k_scale, v_scale, o, lse, B, H, H, N, d, alpha,
                        causal, stream);
}

fa_status fa_fwd_fp8_gqa(const uint8_t *q8, const uint8_t *k8, const uint8_t *v8,
                         const float *q_scale, const float *k_scale, const float *v_scale,
                         void *o, float *lse, int B, int H, int H_kv, int N, int d,
                         float alpha, int causal, void *stream) {
    return fwd_fp8_impl(q8, k8, v8, q_scale, k_scale, v_scale, o, lse, B, H, H_kv, N, d, alpha,
                        causal, stream);
}

// The backward with the causal flag or, with win set, a local window
// (wl, wr); sinks / dsinks (window path only) give the sink logits'
// gradient.
static fa_status bwd_impl(const void *q, const void *k, const void *v, const void *o,
                          const void *dout, const float *lse, float *workspace, void *dq,
                          void *dk, void *dv, int B, int H, int H_kv, int N, int d, float alpha,
                          int causal, bool win, int wl, int wr, float softcap,
                          const float *sinks, float *dsinks, fa_dtype dtype, void *stream) {
    // ---- host-side validation: nothing is launched on failure ----
    if (!q || !k || !v || !o || !dout || !lse || !workspace || !dq || !dk || !dv)
        return FA_ERR_INVALID_ARG;
    if (win && (wl < -1 || wr < -1)) return FA_ERR_INVALID_ARG;
    if (H_kv < 1 || H % H_kv != 0) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(softcap) || softcap < 0.f) return FA_ERR_INVALID_ARG;
    const double cap_pre = softcap > 0.f ? static_cast<double>(alpha) / softcap : 0.0;
    if (!std::isfinite(static_cast<float>(cap_pre))) return FA_ERR_INVALID_ARG;
    if (dsinks && !sinks) return FA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(sinks) & 3u) || (reinterpret_cast<uintptr_t>(dsinks) & 3u))
        return FA_ERR_MISALIGNED;
    if (B < 1 || H < 1 || N < 1 || d < 1) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(alpha)) return FA_ERR_INVALID_ARG;
    if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) ||
        !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
        return FA_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(lse) & 3u) || !aligned16(workspace))
        return FA_ERR_MISALIGNED;
    const uint64_t batch_stride = 2ull * d * H * static_cast<uint64_t>(N);
    if (batch_stride >= (1ull << 40)) return FA_ERR_TOO_LARGE;
    const uint64_t n_t = (static_cast<uint64_t>(N) + 127) / 128;
    const uint64_t units = static_cast<uint64_t>(B) * H * n_t;
    const uint64_t rows = static_cast<uint64_t>(B) * H * N;
    if (units > 0x7fffffffull || rows > 0x7fffffffffffull) return FA_ERR_TOO_LARGE;

    DeviceInfo *dev = nullptr;
    fa_status st = get_device(&dev);
    if (st != FA_OK) return st;

    fa::BwdLaunch L;
    std::memset(&L, 0, sizeof(L));
    const CUtensorMapDataType dt =
        dtype == FA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    if ((st = encode_bshd(&L.q, q, dt, B, H, N, d, 128)) != FA_OK) return st;
    if ((st = encode_bshd(&L.k, k, dt, B, H_kv, N, d, 128)) != FA_OK) return st;
    if ((st = encode_bshd(&L.v, v, dt, B, H_kv, N, d, 128)) != FA_OK) return st;
    if ((st = encode_bshd(&L.dout, dout, dt, B, H, N, d, 128)) != FA_OK) return st;
    L.args.lse = lse;
    L.args.ws_d = workspace;
    L.args.ws_l = workspace + static_cast<size_t>(B) * H * n_t * 128;
    L.args.NP = static_cast<int>(n_t * 128);
    L.args.o = o;
    L.args.dout = dout;
    L.args.dq = dq;
    L.args.dk = dk;
    L.args.dv = dv;
    L.args.status = dev->status;
    L.args.B = B;
    L.args.H = H;
    L.args.N = N;
    L.args.n_t = static_cast<int>(n_t);
    L.args.n_units = static_cast<int>(units);
    const uint64_t units_kv = static_cast<uint64_t>(B) * H_kv * n_t;
    L.args.n_units_kv = static_cast<int>(units_kv);
    L.args.group = H / H_kv;
    L.grid_kv = static_cast<int>(units_kv < static_cast<uint64_t>(dev->sm_count) ? units_kv
                                                                                 : dev->sm_count);
    L.args.scale_log2 = static_cast<float>(static_cast<double>(alpha) * 1.4426950408889634);
    L.args.alpha = alpha;
    L.grid = static_cast<int>(units < static_cast<uint64_t>(dev->sm_count) ? units : dev->sm_count);
    // preprocess: 8 warps per CTA, each warp 4 passes of 32*8/d rows
    const uint64_t rows_per_cta = 8ull * 4ull * (256ull / static_cast<uint64_t>(d));
    const uint64_t gd = (rows + rows_per_cta - 1) / rows_per_cta;
    const uint64_t gcap = 8ull * static_cast<uint64_t>(dev->sm_count);
    L.grid_delta = static_cast<int>(gd < gcap ? gd : gcap);
    L.d = d;
    L.causal = causal != 0;
    L.bf16 = dtype == FA_BF16;
    L.stream = static_cast<cudaStream_t>(stream);
    L.args.wl = wl;
    L.args.wr = wr;
    L.args.sc_pre = static_cast<float>(cap_pre);
    L.args.sc_post = static_cast<float>(static_cast<double>(softcap) * 1.4426950408889634);
    if (causal && !win) {
        // (chunk shares wl's storage: set only here, where no window is read)
        // the forward's dynamic order (set_dynamic_order): one CTA per unit in
        // both main kernels, groups of heads whose streamed inputs (K and V
        // for dQ, Q and dO for dK/dV) fit 32 MiB
        L.grid = static_cast<int>(units);
        L.grid_kv = static_cast<int>(units_kv);
        const uint64_t per_head = 4ull * static_cast<uint64_t>(N) * d;
        uint64_t c = (32ull << 20) / per_head;
        const uint64_t bh = static_cast<uint64_t>(B) * H;
        if (c < 1) c = 1;
        if (c > bh) c = bh;
        L.args.chunk = static_cast<int>(c);
    }
    cudaError_t e = softcap > 0.f ? fa::launch_bwd_win_softcap(L)
                    : win         ? fa::launch_bwd_win(L)
                                  : fa::launch_bwd(L);
    if (e == cudaSuccess && dsinks) e = fa::launch_bwd_dsink(L.args, sinks, dsinks, L.stream);
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout,
                 const float *lse, float *workspace, void *dq, void *dk, void *dv, int B, int H,
                 int N, int d, float alpha, int causal, fa_dtype dtype, void *stream) {
    return bwd_impl(q, k, v, o, dout, lse, workspace, dq, dk, dv, B, H, H, N, d, alpha, causal,
                    false, -1, -1, 0.f, nullptr, nullptr, dtype, stream);
}

fa_status fa_bwd_ext(const void *q, const void *k, const void *v, const void *o,
                     const void *dout, const float *lse, float *workspace, void *dq, void *dk,
                     void *dv, int B, int H, int H_kv, int N, int d, float alpha,
                     int window_left, int window_right, float softcap, const float *sinks,
                     float *dsinks, fa_dtype dtype, void *stream) {
    return bwd_impl(q, k, v, o, dout, lse, workspace, dq, dk, dv, B, H, H_kv, N, d, alpha, 0, true,
                    window_left, window_right, softcap, sinks, dsinks, dtype, stream);
}

// fa_bwd_noalloc: fa_bwd with the workspace taken from the library's own
// device array (g_noalloc_workspace, declared at the top of this file).
fa_status fa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                         const void *dout, const float *lse, void *dq, void *dk, void *dv, int B,
                         int H, int N, int d, float alpha, int causal, fa_dtype dtype,
                         void *stream) {
    // The arguments fa_bwd would reject come first, so the codes match
    // fa_bwd's; only then the limit of the library's array.
    if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || N < 1 || d < 1) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(alpha)) return FA_ERR_INVALID_ARG;
    if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    const uint64_t need = 2ull * B * H * ((static_cast<uint64_t>(N) + 127) / 128) * 128;
    if (need > kNoallocWorkspaceFloats) return FA_ERR_TOO_LARGE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
    float *ws = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (g_noalloc_ptr[dev] == nullptr) {
            // this device is current: its copy of the array
            float *p = nullptr;
            if (cudaGetSymbolAddress(reinterpret_cast<void **>(&p), g_noalloc_workspace) !=
                    cudaSuccess || p == nullptr)
                return FA_ERR_CUDA;
            g_noalloc_ptr[dev] = p;
        }
        ws = g_noalloc_ptr[dev];
    }
    return fa_bwd(q, k, v, o, dout, lse, ws, dq, dk, dv, B, H, N, d, alpha, causal, dtype,
                  stream);
}

fa_status fa_check_status(void *stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
    DeviceInfo *dev = nullptr;
    fa_status st = get_device(&dev);
    if (st != FA_OK) return st;
    uint32_t h[4] = {0, 0, 0, 0};
    if (cudaMemcpy(h, dev->status, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess)
        return FA_ERR_CUDA;
    if (h[0] == 0) return FA_OK;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        std::memcpy(g_last_detail, h, sizeof(h));
    }
    const uint32_t zero[4] = {0, 0, 0, 0};
    if (cudaMemcpy(dev->status, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
        return FA_ERR_CUDA;
    return FA_ERR_TIMEOUT;
}

fa_status fa_selftest_wait_timeout(uint32_t *result, void *stream) {
    if (!result) return FA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(result) & 3u) return FA_ERR_MISALIGNED;
    DeviceInfo *dev = nullptr;
    fa_status st = get_device(&dev);
    if (st != FA_OK) return st;
    cudaError_t e = fa::launch_selftest_timeout(dev->status, result,
                                                static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

void fa_status_detail(uint32_t out[4]) {
    std::lock_guard<std::mutex> lk(g_mu);
    std::memcpy(out, g_last_detail, sizeof(g_last_detail));
}

}  // extern "C"
