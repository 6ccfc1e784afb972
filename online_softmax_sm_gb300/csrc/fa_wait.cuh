// fa_wait.cuh -- bounded mbarrier waits shared by the kernels.  Every wait
// gives up after a global-timer limit: it then sets the CTA's abort flag and
// the device status word (kDevTimeout), and the caller stops cleanly.
#pragma once

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

struct WaitCtx {
  volatile int* abort;
  int* status;
  unsigned long long timeout_ns;
};

// Bounded wait on a phase; false if the CTA aborted or the limit ran out.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const WaitCtx& w) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*w.abort) return false;
    if (global_timer_ns() - t0 > w.timeout_ns) {
      *w.abort = 1;
      atomicExch(w.status, kDevTimeout);
      return false;
    }
  }
}

// Warp-uniform bounded wait: true only if every lane saw the phase complete.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtx& w) {
  return __all_sync(0xffffffffu, wait_bounded(bar, parity, w));
}

// Bounded wait for this thread's own copies / MMAs in flight (ignores abort).
__device__ __forceinline__ void wait_own(uint32_t bar, uint32_t parity,
                                         unsigned long long timeout_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > timeout_ns) return;
  }
}

}  // namespace fa
