// fa_bwd_softcap.cu -- the backward of a forward with a tanh softcap
// ("03 FA3", sec. 5), with or without a local window: both kernels recompute
// t = tanh(alpha s / c) and multiply dS by 1 - t^2.
#include "fa_bwd_launch.cuh"

namespace fa {

cudaError_t launch_bwd_win_softcap(const BwdLaunch &L) {
    if (L.d == 64)
        return L.bf16 ? launch_bwd_inst<64, false, true, true, true>(L)
                      : launch_bwd_inst<64, false, false, true, true>(L);
    return L.bf16 ? launch_bwd_inst<128, false, true, true, true>(L)
                  : launch_bwd_inst<128, false, false, true, true>(L);
}

}  // namespace fa
