// Instantiations of the attention forward kernel for head dim 64.
#include "fa_launch.cuh"

namespace fa {
cudaError_t launch_fwd_d64(const FwdLaunch &L) { return launch_fwd_dispatch<64>(L); }
}  // namespace fa
