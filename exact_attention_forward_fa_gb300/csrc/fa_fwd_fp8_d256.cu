// Instantiations of the FP8 (e4m3 in, bf16 out) one-Q-tile attention forward
// kernel at head dim 256.
#include "fa_launch.cuh"

namespace fa {
cudaError_t launch_fwd_fp8_d256(const FwdLaunch &L) {
    return L.causal ? launch_fwd_fp8_1q_inst<256, true>(L) : launch_fwd_fp8_1q_inst<256, false>(L);
}
}  // namespace fa
