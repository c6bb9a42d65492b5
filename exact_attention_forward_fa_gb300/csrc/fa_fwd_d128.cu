// Instantiations of the attention forward kernel for head dim 128.
#include "fa_launch.cuh"

namespace fa {
cudaError_t launch_fwd_d128(const FwdLaunch &L) { return launch_fwd_dispatch<128>(L); }
}  // namespace fa
