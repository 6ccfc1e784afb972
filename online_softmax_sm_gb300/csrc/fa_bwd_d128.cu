// fa_bwd_d128.cu -- instantiation of the attention backward for head dim 128.
#include "fa_bwd_kernel.cuh"

namespace fa {

cudaError_t launch_bwd_d128(const CUtensorMap* maps, const BwdParams& p, const BwdPreParams& pre,
                           cudaStream_t s) {
  return launch_bwd_t<128>(maps, p, pre, s);
}

}  // namespace fa
