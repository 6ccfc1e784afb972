// Instantiation of the FP8 (E4M3) attention forward: head dim 128, K/V tile 128.
#include "fa_fwd_kernel.cuh"

namespace fa {

cudaError_t launch_fwd_fp8_d128(int qt, const CUtensorMap* maps, const FwdParams& p, dim3 grid,
                                cudaStream_t s) {
  return qt == 2 ? launch_fwd_t<128, 128, 2, true>(maps, p, grid, s)
                 : launch_fwd_t<128, 128, 1, true>(maps, p, grid, s);
}

}  // namespace fa
