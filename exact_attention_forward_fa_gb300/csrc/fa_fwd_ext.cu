// Instantiations of the attention forward kernel with the mask variants:
// local windows and sinks.
#include "fa_launch.cuh"

namespace fa {
cudaError_t launch_fwd_ext(const FwdLaunch &L) {
    return L.d64 ? launch_fwd_ext_dispatch<64, 1>(L) : launch_fwd_ext_dispatch<128, 1>(L);
}
}  // namespace fa
