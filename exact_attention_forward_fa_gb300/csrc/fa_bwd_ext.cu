// fa_bwd_ext.cu -- the backward for local windows ("FlashAttention-3 on
// Hopper", sec. 7.8: both loop bounds tighten, each key tile visits only the
// query tiles of its band) and the gradient of per-head sink logits.
#include "fa_bwd_launch.cuh"

namespace fa {

cudaError_t launch_bwd_win(const BwdLaunch &L) {
    if (L.d == 64)
        return L.bf16 ? launch_bwd_inst<64, false, true, true>(L)
                      : launch_bwd_inst<64, false, false, true>(L);
    return L.bf16 ? launch_bwd_inst<128, false, true, true>(L)
                  : launch_bwd_inst<128, false, false, true>(L);
}

// A sink sigma joins every row's softmax with no value, so its probability
// is P_i = exp(sigma - LSE_i) and its score gradient P_i (0 - D_i); the
// logit's gradient sums that over the rows of every batch.  One CTA per head
// reduces in a fixed order (thread partials, then a tree), so the result is
// the same on every run.  Workspace padding rows have LSE2 = +inf: P = 0.
__global__ void __launch_bounds__(512)
fa_bwd_dsink_kernel(const BwdArgs a, const float *sinks, float *dsinks) {
    const int h = blockIdx.x;
    const float sg = sinks[h] * 1.44269504088896340736f;
    // Each thread walks a fixed set of float4 groups of the padded rows
    // (NP is a multiple of 128; padding rows give 2^-inf * 0 = 0).
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const int n4 = a.NP / 4;
    for (int b = 0; b < a.B; ++b) {
        const size_t base = (static_cast<size_t>(b) * a.H + h) * a.NP;
        const float4 *l4 = reinterpret_cast<const float4 *>(a.ws_l + base);
        const float4 *d4 = reinterpret_cast<const float4 *>(a.ws_d + base);
#pragma unroll 4
        for (int i = threadIdx.x; i < n4; i += blockDim.x) {
            const float4 l = __ldg(l4 + i), dd = __ldg(d4 + i);
            acc[0] = fmaf(-ex2_approx(sg - l.x), dd.x, acc[0]);
            acc[1] = fmaf(-ex2_approx(sg - l.y), dd.y, acc[1]);
            acc[2] = fmaf(-ex2_approx(sg - l.z), dd.z, acc[2]);
            acc[3] = fmaf(-ex2_approx(sg - l.w), dd.w, acc[3]);
        }
    }
    __shared__ float part[512];
    part[threadIdx.x] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
    __syncthreads();
    for (int s = 256; s > 0; s >>= 1) {
        if (threadIdx.x < s) part[threadIdx.x] += part[threadIdx.x + s];
        __syncthreads();
    }
    if (threadIdx.x == 0) dsinks[h] = part[0];
}

cudaError_t launch_bwd_dsink(const BwdArgs &a, const float *sinks, float *dsinks,
                             cudaStream_t stream) {
    fa_bwd_dsink_kernel<<<a.H, 512, 0, stream>>>(a, sinks, dsinks);
    return cudaGetLastError();
}

}  // namespace fa
