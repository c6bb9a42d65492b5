/*
 * fa.h -- C ABI of libfa: exact attention forward for NVIDIA GB300 (sm_103a).
 *
 * The operation ("FlashAttention-3 on Hopper", sec. 3.1 and 4.1-4.7; the
 * Blackwell schedule in "FlashAttention v1-v4", FA4 sections):
 *
 *     S = alpha * Q K^T  (+ causal mask: key j hidden from query i when
 *                          j > i, i.e. col > row + (Nk - Nq) with Nq = Nk)
 *     O = softmax_rows(S) V
 *     LSE_i = log sum_j exp(S_ij)                    (natural log)
 *
 * computed tile by tile with an online softmax, so the N x N score matrix
 * never reaches device memory.  Rows with no visible key would give O = 0,
 * LSE = -inf ("FlashAttention-3 on Hopper", sec. 4.6); with Nq = Nk every
 * row sees at least one key.
 *
 * Layouts (all contiguous, row-major):
 *     Q, K, V, O : [B][N][H][d]   (batch, sequence, head, head dim),
 *                                 element (b,n,h,c) at ((b*N + n)*H + h)*d + c
 *     LSE        : [B][H][N]      float32, element (b,h,n) at (b*H + h)*N + n
 *     FP8 scales : [B][H][ceil(N/128)] float32, one per 128-row tile of a head
 *
 * Conventions for every entry point:
 *   * Pointers named q, k, v, o, lse, x, x8, *_scale are DEVICE pointers
 *     owned by the caller; the library never frees or keeps them.
 *   * `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are asynchronous: they validate, launch and return.
 *   * Arguments are validated on the host before anything is launched; a
 *     failed check returns an error code and launches nothing.
 *   * The library allocates no device memory per call.  It owns one small
 *     per-device status word in a static __device__ variable that kernels
 *     set when a bounded wait gives up; fa_check_status reads it.
 *   * Results are deterministic for fixed inputs: fixed reduction order, no
 *     atomics on outputs.
 *   * Thread safety: entry points may be called from several host threads;
 *     the per-device caches inside are guarded by a mutex.
 */
#ifndef FA_H_
#define FA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size, bad flag, non-finite alpha */
    FA_ERR_UNSUPPORTED = 2,  /* head dim or dtype without a kernel, or not an sm_103 device */
    FA_ERR_MISALIGNED = 3,   /* a tensor pointer is not 16-byte aligned (TMA rule) */
    FA_ERR_TOO_LARGE = 4,    /* a size exceeds the TMA descriptor limits */
    FA_ERR_CUDA = 5,         /* a CUDA runtime/driver call or the launch failed */
    FA_ERR_TIMEOUT = 6       /* a kernel's bounded wait gave up (fa_check_status) */
} fa_status;

typedef enum {
    FA_BF16 = 0,
    FA_FP16 = 1
} fa_dtype;

/* Scale granularity of the FP8 pre-pass (fa_quantize_fp8_granular). */
typedef enum {
    FA_SCALE_TILE = 0,    /* one scale per 128-row tile of a head (block quantization) */
    FA_SCALE_HEAD = 1,    /* one scale per (batch, head) */
    FA_SCALE_TENSOR = 2   /* one scale for the whole tensor */
} fa_scale_granularity;

/*
 * fa_fwd -- exact attention forward, BF16 or FP16 in and out.
 *   q, k, v : device, [B][N][H][d] in `dtype`, 16-byte aligned.
 *   o       : device, [B][N][H][d] in `dtype`, 16-byte aligned (written).
 *   lse     : device, float [B][H][N], 4-byte aligned, or NULL to skip.
 *   B, H, N : >= 1.  d in {64, 128, 256}; other head dims return
 *             FA_ERR_UNSUPPORTED.
 *   alpha   : the score scale (usually 1/sqrt(d)); must be finite.
 *   causal  : 0 or 1.
 * Accumulation is FP32; P is rounded to `dtype` before the P V product and
 * the softmax denominator sums those same rounded values; O is rounded to
 * `dtype` round-to-nearest-even.
 * Causal launches have one CTA per work unit and let running CTAs take over
 * those not yet started (cluster launch control), in an order that keeps
 * groups of heads together for L2 reuse of K and V; which CTA computes a
 * tile varies from launch to launch, the results do not.
 */
fa_status fa_fwd(const void *q, const void *k, const void *v, void *o,
                 float *lse, int B, int H, int N, int d, float alpha,
                 int causal, fa_dtype dtype, void *stream);

/*
 * fa_fwd_gqa -- fa_fwd with grouped key/value heads (grouped-query and
 * multi-query attention: "FlashAttention-3 on Hopper", ch. 11 and the GQA
 * remark of sec. 7.2.3): q, o are [B][N][H][d] as in fa_fwd, k, v are
 * [B][N][H_kv][d], H_kv >= 1 divides H, and query head h attends with key /
 * value head h / (H / H_kv).  H_kv = H is fa_fwd; H_kv = 1 is multi-query
 * attention.  H % H_kv != 0 or H_kv < 1 returns FA_ERR_INVALID_ARG; other
 * arguments, results and errors as fa_fwd.
 */
fa_status fa_fwd_gqa(const void *q, const void *k, const void *v, void *o,
                     float *lse, int B, int H, int H_kv, int N, int d,
                     float alpha, int causal, fa_dtype dtype, void *stream);

/*
 * fa_fwd_gqa_packed -- fa_fwd_gqa with the g = H / H_kv query heads of each
 * key/value head packed into the rows of one Q tile ("PackGQA" of the GQA
 * remark in "FlashAttention-3 on Hopper"): a tile holds 128 / g query
 * positions of all g heads, so one pass over a key/value head's K and V
 * serves the whole group and short sequences do not leave tiles half
 * empty.  Same arguments, layouts, results (up to FP32 rounding order: the
 * softmax's rescale decisions are taken per warp of rows) and errors as
 * fa_fwd_gqa; additionally d must be 64 or 128 and g must divide 128
 * (g = 1 runs fa_fwd_gqa), else FA_ERR_UNSUPPORTED.  Measured on GB300
 * (H 32 over H_kv 2 or 8, d 128): N = 64 twice the throughput of
 * fa_fwd_gqa, N = 256 about the same, N = 4096 2-5 % below it -- a choice
 * for short sequences.
 */
fa_status fa_fwd_gqa_packed(const void *q, const void *k, const void *v, void *o,
                            float *lse, int B, int H, int H_kv, int N, int d,
                            float alpha, int causal, fa_dtype dtype, void *stream);

/*
 * fa_fwd_ext -- fa_fwd_gqa with the score and mask variants of
 * "FlashAttention-3 on Hopper" sec. 4.6 (learnable sinks folded into the
 * row sum at finalize) and sec. 4.7 (local / sliding-window masks; a score
 * transformation precedes the mask), and the softcap of "03 FA3" sec. 5:
 *   window_left, window_right : key j is hidden from query i when
 *            j > i + window_right (window_right >= 0) or
 *            j < i - window_left (window_left >= 0); -1 = no bound on that
 *            side.  (-1, 0) is causal, (-1, -1) no mask; values below -1
 *            return FA_ERR_INVALID_ARG.  Every row sees at least key i.
 *   softcap : 0 for none, else c > 0: each visible score s = alpha q.k
 *            becomes c tanh(s / c) before the mask and the softmax
 *            (tanh.approx.f32: max abs error 8e-6, measured);
 *            negative or non-finite returns FA_ERR_INVALID_ARG.
 *   sinks  : device, float [H] (one logit sigma per query head, finite or
 *            -inf), 4-byte aligned, or NULL for none.  sigma joins every
 *            row's softmax denominator and carries no value:
 *            O_i = sum_j e^(S_ij) v_j / (sum_j e^(S_ij) + e^sigma),
 *            LSE_i = log(sum_j e^(S_ij) + e^sigma).
 *   d in {64, 128} (others FA_ERR_UNSUPPORTED).  Other arguments, results
 *   and errors as fa_fwd_gqa.  Key tiles entirely outside a Q tile's
 *   window are neither loaded nor computed.
 */
fa_status fa_fwd_ext(const void *q, const void *k, const void *v, void *o,
                     float *lse, int B, int H, int H_kv, int N, int d,
                     float alpha, int window_left, int window_right,
                     float softcap, const float *sinks, fa_dtype dtype,
                     void *stream);

/*
 * fa_fwd_splitkv -- fa_fwd with each work unit's key range cut into
 * n_splits parts ("FlashAttention-3 on Hopper", ch. 10: split-KV and its
 * combine kernel), for problems whose B * H * ceil(N/256) units do not
 * fill the GPU.  Every split writes its partial O (FP32, normalised over
 * its own keys) and LSE into `workspace`; a combine kernel then writes
 *   LSE = log sum_s exp(LSE_s),  O = sum_s exp(LSE_s - LSE) O_s
 * to o (dtype) and lse (if not NULL).
 *   workspace : device, fa_splitkv_workspace_floats(B, H, N, d, n_splits)
 *            floats, 16-byte aligned, caller-owned; nothing in it needs to
 *            start at zero.
 *   n_splits in [1, 16] (FA_ERR_INVALID_ARG otherwise); d in {64, 128}
 *   (others FA_ERR_UNSUPPORTED).  Other arguments and errors as fa_fwd.
 */
fa_status fa_fwd_splitkv(const void *q, const void *k, const void *v, void *o,
                         float *lse, int B, int H, int N, int d, float alpha,
                         int causal, fa_dtype dtype, int n_splits,
                         float *workspace, void *stream);

/* fa_splitkv_workspace_floats -- workspace size of fa_fwd_splitkv, in
 * floats: n_splits * (B*N*H*d + B*H*N); -1 for a non-positive argument. */
long long fa_splitkv_workspace_floats(int B, int H, int N, int d, int n_splits);

/* fa_splitkv_auto -- a split count for the current device: with
 * u = B * H * ceil(ceil(N/128)/2) work units, 1 when u already occupies 80 %
 * of the SMs, else the fewest splits S with S u >= 80 % of the SMs, keeping
 * S u within one wave, at least 4 key tiles per split and S <= 16. */
int fa_splitkv_auto(int B, int H, int N, int d);

/*
 * fa_quantize_fp8 -- FP8 pre-pass: block quantization with optional
 * incoherent processing ("FlashAttention-3 on Hopper", sec. 6.3 and 6.4).
 *   x      : device, bf16 [B][N][H][d], 16-byte aligned.
 *   x8     : device, uint8 e4m3 codes [B][N][H][d], 16-byte aligned (written).
 *   scales : device, float [B][H][ceil(N/128)] (written): one scale per
 *            128-row tile of a head, scale = amax / 448 over the (rotated)
 *            tile, 1 for an all-zero tile.
 *   hadamard_signs : device, float[d] of +-1, or NULL for no rotation.  With
 *            it, each row is replaced by y = x (1/sqrt d) H D before
 *            quantization (H: d x d Sylvester Hadamard matrix, D = diag of
 *            the signs).  Use the same signs for Q and K, none for V: the
 *            product (QM)(KM)^T equals Q K^T because M is orthogonal.
 *   d in {64, 128, 256}.
 * codes = e4m3(y * (1/scale)) with the FP32 reciprocal formed once per tile
 * (within one rounding of y / scale), round to nearest even, saturating at
 * +-448.
 */
fa_status fa_quantize_fp8(const void *x, uint8_t *x8, float *scales,
                          const float *hadamard_signs, int B, int H, int N, int d,
                          void *stream);

/*
 * fa_quantize_fp8_granular -- fa_quantize_fp8 with a coarser scale: the
 * control arm of the FA3 FP8 numerical-error ablation, which compares block
 * quantization against one scale per tensor (the FlashAttention-3 review on
 * diycv.top, "numerical error"; "FlashAttention-3 on Hopper", sec. 6.3).
 *   granularity : FA_SCALE_TILE (exactly fa_quantize_fp8), FA_SCALE_HEAD
 *            (scale = amax / 448 over each (b, h)), or FA_SCALE_TENSOR (over
 *            the whole tensor); other values give FA_ERR_INVALID_ARG.
 *   scales : written in the per-tile layout [B][H][ceil(N/128)] whatever
 *            the granularity (every tile of a group holds the group's
 *            scale), so fa_fwd_fp8 consumes them unchanged.
 * Coarser granularities run three kernels on `stream` (the per-tile pass,
 * a maximum over each group of its tile scales, and the pass again with
 * those scales).  Other arguments, results and errors as fa_quantize_fp8.
 */
fa_status fa_quantize_fp8_granular(const void *x, uint8_t *x8, float *scales,
                                   const float *hadamard_signs, int B, int H, int N,
                                   int d, int granularity, void *stream);

/*
 * fa_fwd_fp8 -- attention forward on e4m3 Q/K/V with per-tile scales
 * (as written by fa_quantize_fp8), bf16 output ("FlashAttention-3 on
 * Hopper", sec. 6.3: descales folded into the softmax scale per tile
 * pair; "03 FA3", sec. 4: the exponent of the FP8 probabilities shifted
 * into the e4m3 range: P' = 2^(s - r + c) with the reference r moved when
 * a tile's row max exceeds it by more than tau; c = 4, tau = 4.8, so
 * P' <= 2^8.8 < 448: the pages' c = 8 would leave tau = 0.8 and a rescale
 * on about half of the steps of outlier inputs).
 *   q8, k8, v8 : device, uint8 e4m3 [B][N][H][d], 16-byte aligned.
 *   q_scale, k_scale, v_scale : device, float [B][H][ceil(N/128)].
 *   o   : device, bf16 [B][N][H][d] (written).  lse : as for fa_fwd.
 *   d in {128, 256} (others return FA_ERR_UNSUPPORTED; d = 256 runs one
 *   128-row Q tile per work unit).  alpha, causal as fa_fwd.
 * P is rounded to e4m3 before the P V product with the V tile scale
 * folded in (P'_j = P_j v_j / max_j v_j); accumulation is FP32, and O is
 * normalised by the FP32 row sum of the unrounded P.  Per-tile V scales
 * are accepted, but the fold then rounds the dominant terms of P' (ratios
 * below 1 are not powers of two), which the row sum does not see; one V
 * scale per head (fa_quantize_fp8_granular with FA_SCALE_HEAD, repeated
 * over the tiles) makes every ratio 1 and is the measured better choice.
 */
fa_status fa_fwd_fp8(const uint8_t *q8, const uint8_t *k8, const uint8_t *v8,
                     const float *q_scale, const float *k_scale, const float *v_scale,
                     void *o, float *lse, int B, int H, int N, int d, float alpha,
                     int causal, void *stream);

/*
 * fa_fwd_fp8_gqa -- fa_fwd_fp8 with grouped key/value heads (as fa_fwd_gqa):
 * q8 and q_scale have H heads, k8, v8, k_scale and v_scale have H_kv heads
 * ([B][N][H_kv][d] codes, [B][H_kv][ceil(N/128)] scales), H_kv >= 1 divides
 * H, and query head h attends with key/value head h / (H / H_kv).  H_kv = H
 * is fa_fwd_fp8.  H % H_kv != 0 or H_kv < 1 returns FA_ERR_INVALID_ARG;
 * other arguments, results and errors as fa_fwd_fp8.
 */
fa_status fa_fwd_fp8_gqa(const uint8_t *q8, const uint8_t *k8, const uint8_t *v8,
                         const float *q_scale, const float *k_scale, const float *v_scale,
                         void *o, float *lse, int B, int H, int H_kv, int N, int d,
                         float alpha, int causal, void *stream);

/*
 * fa_bwd -- gradients of the attention of fa_fwd ("FlashAttention-3 on
 * Hopper", ch. 7): with S = alpha Q K^T (masked as in fa_fwd),
 * P = softmax(S) and O = P V, for the upstream gradient dO:
 *   dV = P^T dO,  dP = dO V^T,  D_i = rowsum(dO_i o O_i),
 *   dS = P o (dP - D),  dQ = alpha dS K,  dK = alpha dS^T Q.
 * P is recomputed from Q, K and the forward's LSE (sec. 7.1.3).
 *   q, k, v, o, dout : device, dtype [B][N][H][d], 16-byte aligned; o and
 *            lse are the outputs of fa_fwd on the same q, k, v, alpha and
 *            causal.
 *   lse    : device, float [B][H][N] (natural log, as fa_fwd writes it).
 *   workspace : device, float [2][B][H][ceil(N/128)*128], 16-byte aligned,
 *            caller-owned; receives D = rowsum(dO o O) and LSE*log2(e) per
 *            row (rows padded to whole 128-row tiles).
 *   dq, dk, dv : device, dtype [B][N][H][d], 16-byte aligned (written).
 *   d in {64, 128} (others return FA_ERR_UNSUPPORTED); alpha, causal,
 *   dtype and stream as fa_fwd.
 * Three kernels run in order on `stream`: the D preprocess, a key-parallel
 * kernel for dK and dV and a query-parallel kernel for dQ that recomputes S
 * and dP (sec. 7.2, first option), so no atomics are used and the results
 * are identical from run to run.  P and dS are rounded to `dtype` for the
 * GEMMs that consume them; accumulation is FP32; outputs are rounded to
 * `dtype`.  Nothing is allocated.  Errors as fa_fwd.  With causal = 1 both
 * main kernels schedule their units as fa_fwd's causal launches do (one CTA
 * per unit, head groups kept together for L2 reuse).
 */
fa_status fa_bwd(const void *q, const void *k, const void *v, const void *o,
                 const void *dout, const float *lse, float *workspace, void *dq,
                 void *dk, void *dv, int B, int H, int N, int d, float alpha,
                 int causal, fa_dtype dtype, void *stream);

/*
 * fa_bwd_ext -- fa_bwd for the forward of fa_fwd_ext with a local window,
 * an optional softcap and optional sinks ("FlashAttention-3 on Hopper",
 * sec. 7.8: a right window bounds the first query tile a key tile visits, a
 * left window the last, and the softcap enters as a score modifier; sec.
 * 4.6: sinks; "03 FA3", sec. 5: softcap).
 *   window_left, window_right : as for fa_fwd_ext (-1 = no bound; values
 *            below -1 return FA_ERR_INVALID_ARG).
 *   softcap : the forward's c (0: none).  With c > 0 both kernels recompute
 *            t = tanh(alpha s / c) (tanh.approx.f32), form P from t and the
 *            LSE, and scale dS by dS/du = 1 - t^2.  Negative, non-finite or
 *            alpha / c beyond FP32 returns FA_ERR_INVALID_ARG.
 *   lse    : from fa_fwd_ext with the same window and sinks.  The gradients
 *            of q, k and v need nothing else from the sinks: P is formed
 *            from that LSE, which already holds the sink term.
 *   sinks  : device float [H] (the forward's), or NULL.  dsinks : device
 *            float [H] or NULL; with both, dsinks[h] receives the gradient
 *            of sigma_h, -sum over batches and rows of e^(sigma_h - LSE) D
 *            (D = rowsum(dO o O)), reduced in a fixed order.  dsinks
 *            without sinks returns FA_ERR_INVALID_ARG.
 *   H_kv   : K/V heads (grouped-query attention, as for fa_fwd_ext): k, v,
 *            dk, dv are [B][N][H_kv][d], query head h uses K/V head
 *            h / (H / H_kv), and dK, dV of a K/V head sum the contributions
 *            of all its query heads (accumulated in FP32 in one kernel, no
 *            atomics).  H % H_kv != 0 or H_kv < 1 returns FA_ERR_INVALID_ARG.
 * Other arguments, results and errors as fa_bwd (d in {64, 128}).
 */
fa_status fa_bwd_ext(const void *q, const void *k, const void *v, const void *o,
                     const void *dout, const float *lse, float *workspace,
                     void *dq, void *dk, void *dv, int B, int H, int H_kv, int N, int d,
                     float alpha, int window_left, int window_right,
                     float softcap, const float *sinks, float *dsinks,
                     fa_dtype dtype, void *stream);

/*
 * fa_bwd_noalloc -- fa_bwd without a caller-provided workspace (the pages
 * have no counterpart: this is an interface convenience of this library).
 * For callers that must not allocate device memory at the point of the
 * call, e.g. a program whose device memory is reserved up front or a
 * runtime that forbids allocation inside a step.  The workspace is a
 * 16 MiB array in the library's device image (one per device that loads
 * the library, held until the process exits); nothing is allocated, and
 * nothing in it needs to start at zero.  Limit: 2 * B * H * ceil(N/128) *
 * 128 <= 4194304 floats, else FA_ERR_TOO_LARGE before anything runs; the
 * arguments fa_bwd rejects are checked first and give fa_bwd's codes.
 * Calls that overlap in time (on other streams or host threads) share the
 * array and race; serialise them.  The array's device address is looked up
 * on the first call on each device (with that device current) and cached,
 * so make that first call before any stream capture, and do not call this
 * after a cudaDeviceReset in the same process (the cached address would be
 * stale).  Other arguments, results and errors as fa_bwd.
 */
fa_status fa_bwd_noalloc(const void *q, const void *k, const void *v,
                         const void *o, const void *dout, const float *lse,
                         void *dq, void *dk, void *dv, int B, int H, int N,
                         int d, float alpha, int causal, fa_dtype dtype,
                         void *stream);

/*
 * fa_check_status -- synchronizes `stream`, then reports and clears the
 * device status word of the current device.  Returns FA_ERR_TIMEOUT if a
 * kernel launched since the last check gave up on a bounded wait (its
 * outputs are then undefined), FA_ERR_CUDA if the synchronization failed,
 * FA_OK otherwise.
 */
fa_status fa_check_status(void *stream);

/*
 * fa_status_detail -- the status word captured by the last fa_check_status
 * that returned FA_ERR_TIMEOUT: out[0] code, out[1] role that gave up
 * (1/2 softmax group L/H, 3 producer, 4 MMA issuer, 6 FP8 pre-pass,
 * 7 self-test),
 * out[2] wait site,
 * out[3] block index.  Zeros if no timeout was ever reported.
 */
void fa_status_detail(uint32_t out[4]);

/*
 * fa_selftest_wait_timeout -- exercises the failure path without a fault:
 * one CTA whose two warps wait (with the pipeline kernels' bounded wait) on
 * valid mbarriers that nobody arrives on.  The first wait gives up after
 * its time limit (2 s), records role 7 and its site (1 or 2) in the status
 * word and raises the CTA's abort flag; the other then returns promptly.
 *   result : device, uint32_t[2], 4-byte aligned (written): result[w] = 1
 *            when warp w's wait returned false.
 * The next fa_check_status then returns FA_ERR_TIMEOUT and
 * fa_status_detail gives {1, 7, site, 0}; the CUDA context stays usable.
 * Returns FA_ERR_INVALID_ARG for a null result, FA_ERR_MISALIGNED,
 * FA_ERR_UNSUPPORTED / FA_ERR_CUDA as fa_fwd.
 */
fa_status fa_selftest_wait_timeout(uint32_t *result, void *stream);

/* fa_status_string -- a static, human-readable name for a status code. */
const char *fa_status_string(fa_status s);

/* fa_version -- library version as major*10000 + minor*100 + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
