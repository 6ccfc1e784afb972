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

// Records a failure in the device status word unless one is recorded already
// (the first failure wins).
__device__ __forceinline__ void record_status(int* status, int code) { atomicCAS(status, kDevOk, code); }

// Debug build (FA_DEBUG): FA_DCHECK(cond, status) is true when cond holds;
// otherwise it records kDevCheck and the source line in the status words and
// is false, so the guarded access is skipped (nothing traps).  In the release
// build it is the constant true and costs nothing.
#ifdef FA_DEBUG
__device__ __forceinline__ bool dcheck(bool ok, int* status, int line) {
  if (!ok && atomicCAS(status, kDevOk, kDevCheck) == kDevOk) atomicExch(status + 1, line);
  return ok;
}
#define FA_DCHECK(cond, status) ::fa::dcheck(static_cast<bool>(cond), (status), __LINE__)
#else
#define FA_DCHECK(cond, status) true
#endif

// Bounded wait on a phase; false if the CTA aborted or the limit ran out.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const WaitCtx& w) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*w.abort) return false;
    if (global_timer_ns() - t0 > w.timeout_ns) {
      *w.abort = 1;
      record_status(w.status, kDevTimeout);
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
