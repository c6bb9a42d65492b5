// Instantiations of the attention forward kernel with split key ranges
// (split-KV: partial O and LSE per split, merged by fa_splitkv.cu).
#include "fa_launch.cuh"

namespace fa {
cudaError_t launch_fwd_split(const FwdLaunch &L) {
    // the head dim is carried by the caller's choice of instantiation
    return L.d64 ? launch_fwd_split_dispatch<64>(L) : launch_fwd_split_dispatch<128>(L);
}
}  // namespace fa
