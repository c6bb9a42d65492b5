// Instantiations of the attention forward kernel for head dim 256.
#include "fa_launch.cuh"

namespace fa {
cudaError_t launch_fwd_d256(const FwdLaunch &L) {
    if (L.causal) {
        return L.bf16 ? launch_fwd_1q_inst<256, true, true>(L)
                      : launch_fwd_1q_inst<256, true, false>(L);
    }
    return L.bf16 ? launch_fwd_1q_inst<256, false, true>(L)
                  : launch_fwd_1q_inst<256, false, false>(L);
}
}  // namespace fa
