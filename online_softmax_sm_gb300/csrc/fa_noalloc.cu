// fa_noalloc.cu -- split-KV forward for callers that must not allocate.
//
// Some callers cannot call cudaMalloc (or any allocating routine) on the
// path that runs attention: runtimes without a device allocator, hosts that
// have handed all device memory to their own pool, or latency-bound loops in
// which an allocation could block or synchronise.  fa_fwd with n_splits > 1
// takes its workspace with cudaMallocAsync, so it is unusable there.  This
// entry point runs fa_fwd's own split-KV path (partial kernel, then merge)
// with the workspace in a fixed device array that lives as long as the
// library is loaded.
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "fa_internal.h"

namespace {

// One per device that loads the library, held until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices];  // device address of g_noalloc_scratch, per device

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Device address of the scratch array on the current device.  In host code
// the symbol is only a host-side stand-in, so the address must come from
// cudaGetSymbolAddress, once per device, with that device current.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return FA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return FA_OK;
}

}  // namespace

extern "C" int fa_fwd_split_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                                    int B, int H, int Nq, int Nk, int d, float scale, int causal,
                                    int n_splits, void* stream) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || n_splits < 2 || n_splits > 65535)
    return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(o) & 15) || (reinterpret_cast<uintptr_t>(lse) & 3))
    return FA_ERR_INVALID_ARG;
  // Same split count as fa_fwd: at most one split per K/V tile of the default size.
  const int kv_tiles = (Nk + fa::kDefaultBc - 1) / fa::kDefaultBc;
  const int splits = n_splits < kv_tiles ? n_splits : kv_tiles;
  if (splits < 2) return fa_fwd(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, 1, stream);
  // fa_fwd's split workspace layout: m, l fp32 and O_s in bf16, each 256-byte aligned
  const size_t rows = static_cast<size_t>(B) * H * Nq;
  const size_t ml = align256(static_cast<size_t>(splits) * rows * sizeof(float));
  const size_t need = 2 * ml + align256(static_cast<size_t>(splits) * rows * d * 2);
  if (need > FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_SCRATCH_TOO_SMALL;
  void* base = nullptr;
  int rc = scratch_address(&base);
  if (rc != FA_OK) return rc;
  // Every entry the merge reads is written by the partial kernel first (empty
  // splits write m = -inf, l = 0, O = 0), so nothing has to start at zero.
  return fa::fwd_split_into(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, splits, stream, base,
                            FA_NOALLOC_SCRATCH_BYTES);
}
