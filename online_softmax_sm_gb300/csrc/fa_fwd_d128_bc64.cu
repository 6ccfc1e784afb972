// Instantiation of the attention forward kernel for head dim 128, K/V tile 64.
#include "fa_fwd_kernel.cuh"

namespace fa {

cudaError_t launch_fwd_d128_bc64(int qt, const CUtensorMap* maps, const FwdParams& p, dim3 grid,
                                cudaStream_t s) {
  return qt == 2 ? launch_fwd_t<128, 64, 2>(maps, p, grid, s)
                 : launch_fwd_t<128, 64, 1>(maps, p, grid, s);
}

}  // namespace fa
