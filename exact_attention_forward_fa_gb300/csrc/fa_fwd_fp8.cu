// Instantiations of the FP8 (e4m3 in, bf16 out) attention forward kernel,
// head dim 128.
#include "fa_launch.cuh"

namespace fa {
cudaError_t launch_fwd_fp8(const FwdLaunch &L) {
    return L.causal ? launch_fwd_inst<128, true, true, true>(L)
                    : launch_fwd_inst<128, false, true, true>(L);
}
}  // namespace fa
