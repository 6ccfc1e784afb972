// fa_bwd_d64.cu -- instantiation of the attention backward for head dim 64.
#include "fa_bwd_kernel.cuh"

namespace fa {

cudaError_t launch_bwd_d64(const CUtensorMap* maps, const BwdParams& p, const BwdPreParams& pre,
                           cudaStream_t s) {
  return launch_bwd_t<64>(maps, p, pre, s);
}

}  // namespace fa
