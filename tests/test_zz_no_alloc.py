"""fa_fwd_split_noalloc: the split-KV forward for callers that cannot allocate.

Runtimes without a device allocator, hosts whose device memory belongs to
their own pool, and latency-bound loops where an allocation could block
cannot let the library call cudaMallocAsync the way fa_fwd does for its
split-KV workspace.  This entry point keeps that workspace in a fixed device
array instead.  Checked here through the C ABI against fa_fwd with the same number
of splits, within the parity tolerances, on two calls in a row (the second
with different shapes and inputs, so stale scratch contents would show), and
its size limit is checked to be refused before anything is launched.

Collected last on purpose: a failure here leaves every other test already run.
"""
import ctypes

import pytest
import torch

import online_softmax_sm_gb300 as fa
from online_softmax_sm_gb300 import _binding, workloads
from tests import _parity as P

pytestmark = pytest.mark.gpu


def _noalloc_raw(q, k, v, scale, causal, n_splits):
    """Direct ctypes call of the C entry point (no Python-side checks)."""
    L = fa.lib()
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    rc = L.fa_fwd_split_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                B, H, Nq, Nk, d, ctypes.c_float(scale), int(causal), n_splits,
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc, o, lse


CALLS = [
    # B, H, Nq, Nk, d, causal, n_splits   (workspace well under the fixed limit)
    (2, 4, 128, 5000, 128, False, 8),
    (1, 3, 200, 3000, 64, True, 5),
]


def test_noalloc_matches_fwd_on_two_calls_in_a_row():
    for idx, (B, H, Nq, Nk, d, causal, ns) in enumerate(CALLS):
        assert fa.split_workspace_bytes(B, H, Nq, d, ns) <= _binding.NOALLOC_SCRATCH_BYTES
        w = workloads.custom(B, H, Nq, Nk, d, seed=70 + idx, causal=causal, q_mult=2.0)
        q, k, v = workloads.generate(w, device="cuda")
        rc, o1, l1 = _noalloc_raw(q, k, v, w.scale, causal, ns)
        assert rc == fa.FA_OK, fa.strerror(rc)
        o2, l2 = fa.fwd(q, k, v, w.scale, causal, ns)
        torch.cuda.synchronize()
        assert fa.device_status() == fa.FA_OK
        d_o = (o1.float() - o2.float()).abs()
        assert d_o.max().item() <= P.MAX_ABS_O and d_o.mean().item() <= P.MEAN_ABS_O
        fin = torch.isfinite(l2)
        assert torch.equal(fin, torch.isfinite(l1))
        assert torch.equal(torch.isneginf(l1), torch.isneginf(l2))
        if fin.any():
            assert (l1[fin] - l2[fin]).abs().max().item() <= P.MAX_ABS_LSE
        # same kernels on the same inputs: expected to agree bit for bit
        assert torch.equal(o1, o2)


def test_noalloc_refuses_workspace_over_the_limit():
    # 16 splits of B*H*Nq = 65536 rows at d = 128 need ~545 MB > 32 MiB: refused
    # during argument checks, before any launch (the tiny buffers are never read).
    t = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    l = torch.zeros(16, dtype=torch.float32, device="cuda")
    L = fa.lib()
    rc = L.fa_fwd_split_noalloc(t.data_ptr(), t.data_ptr(), t.data_ptr(), t.data_ptr(), l.data_ptr(),
                                16, 32, 128, 32768, 128, ctypes.c_float(0.088), 0, 16,
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == fa.FA_ERR_SCRATCH_TOO_SMALL
    assert "scratch" in fa.strerror(rc)
