// fa_bwd.cu -- instantiations of the backward kernels (fa_bwd_kernel.cuh)
// for the plain and causal masks.
#include "fa_bwd_launch.cuh"

namespace fa {

cudaError_t launch_bwd(const BwdLaunch &L) {
    if (L.d == 64) {
        if (L.bf16) return L.causal ? launch_bwd_inst<64, true, true>(L) : launch_bwd_inst<64, false, true>(L);
        return L.causal ? launch_bwd_inst<64, true, false>(L) : launch_bwd_inst<64, false, false>(L);
    }
    if (L.bf16) return L.causal ? launch_bwd_inst<128, true, true>(L) : launch_bwd_inst<128, false, true>(L);
    return L.causal ? launch_bwd_inst<128, true, false>(L) : launch_bwd_inst<128, false, false>(L);
}

}  // namespace fa
