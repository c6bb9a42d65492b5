// Instantiations of the attention forward kernel with a softcap on the
// scores (plus local windows and sinks).
#include "fa_launch.cuh"

namespace fa {
cudaError_t launch_fwd_ext_softcap(const FwdLaunch &L) {
    return L.d64 ? launch_fwd_ext_dispatch<64, 2>(L) : launch_fwd_ext_dispatch<128, 2>(L);
}
}  // namespace fa
