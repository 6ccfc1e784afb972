"""Single-pass online-softmax attention forward for GB300 (sm_103a).

The compute path is libfa.so (hand-written CUDA, C ABI in include/fa.h); this
package is its Python binding plus the seeded workload generators:

  fwd(q, k, v, scale, causal, n_splits)   -> (o, lse)       fa_fwd / fa_fwd_ex
  fwd_host(q, k, v, scale, causal)        -> (o, lse)       fa_fwd_host (CPU tensors, copies included)
  fwd_host(..., window=(wl, wr))          -> (o, lse)       fa_fwd_local_host
  fwd_local(q, k, v, wl, wr, ...)         -> (o, lse)       fa_fwd_local (sliding window)
  fwd_fp8(q8, k8, v8, ...)                -> (o, lse)       fa_fwd_fp8 (E4M3, Max_offset 8)
  fwd_fp8_host(q8, k8, v8, ...)           -> (o, lse)       fa_fwd_fp8_host (CPU tensors, copies included)
  bwd_host(q, k, v, o, lse, dout, ...)    -> (dq, dk, dv)   fa_bwd_host / fa_bwd_local_host (CPU tensors)
  fwd_partial(q, k, v, n_splits, ...)     -> (m, l, o) parts fa_fwd_partial
  merge_splits(m_part, l_part, o_part)    -> (o, lse)       fa_merge_splits
  fwd_split_noalloc(q, k, v, n_splits)   -> (o, lse)       fa_fwd_split_noalloc
  softmax_rows(x)                         -> (y, lse)       fa_softmax_rows (two-pass normaliser)
  bwd(q, k, v, o, lse, dout, ...)         -> (dq, dk, dv)   fa_bwd / fa_bwd_local
  split_workspace_bytes(...), device_status(), version()

libfa.so is loaded on first use; importing the package loads nothing.
"""
from ._binding import (FA_DTYPE_BF16, FA_DTYPE_F32, FA_ERR_CUDA, FA_ERR_DEVICE_CHECK, FA_ERR_DEVICE_TIMEOUT,
                       FA_ERR_INVALID_ARG, FA_ERR_NO_MEMORY, FA_ERR_SCRATCH_TOO_SMALL,
                       FA_ERR_UNSUPPORTED, FA_OK, FAError, bwd, bwd_host, debug_library, device_status, fwd, fwd_fp8, fwd_fp8_host, fwd_host, fwd_local,
                       fwd_partial, fwd_split_noalloc, lib, merge_splits, softmax_rows,
                       split_workspace_bytes, strerror, version)

__all__ = ["fwd", "fwd_host", "fwd_local", "fwd_fp8", "fwd_fp8_host", "bwd", "bwd_host", "fwd_partial", "merge_splits", "fwd_split_noalloc", "softmax_rows",
           "split_workspace_bytes", "device_status", "version", "strerror", "lib", "FAError",
           "FA_OK", "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED", "FA_ERR_CUDA",
           "FA_ERR_DEVICE_TIMEOUT", "FA_ERR_DEVICE_CHECK", "debug_library", "FA_ERR_NO_MEMORY", "FA_ERR_SCRATCH_TOO_SMALL", "FA_DTYPE_F32",
           "FA_DTYPE_BF16"]
