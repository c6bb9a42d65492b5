// Instantiations of the attention forward kernel with the query heads of
// one key/value head packed into its Q tiles (grouped heads).
#include "fa_launch.cuh"

namespace fa {
cudaError_t launch_fwd_pack(const FwdLaunch &L) {
    return L.d64 ? launch_fwd_pack_dispatch<64>(L) : launch_fwd_pack_dispatch<128>(L);
}
}  // namespace fa
