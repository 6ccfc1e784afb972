"""Failure detection without a GPU fault.

Every wait inside the kernels is bounded by a global-timer limit.  The test
hook `test_skip_kv_load = n` makes the producer of every CTA skip its n-th
K/V tile load: the consumer's wait for that tile runs out (a flag nothing
sets), the CTA stops cleanly, and the call reports FA_ERR_DEVICE_TIMEOUT
through fa_get_device_status.  The context must stay usable: a normal call
right after still matches the oracle.
"""
import pytest
import torch

import online_softmax_sm_gb300 as fa
from online_softmax_sm_gb300 import workloads
from tests import _parity as P

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,n_splits,skip", [
    (1, 2, 256, 1024, 128, False, 1, 3),   # two Q tiles per CTA, skip V_0
    (1, 2, 128, 1024, 64, False, 1, 1),    # one Q tile per CTA, skip K_0
    (1, 1, 300, 700, 128, True, 3, 2),     # split-KV partials, skip K_1
])
def test_missing_load_times_out_cleanly(B, H, Nq, Nk, d, causal, n_splits, skip):
    w = workloads.custom(B, H, Nq, Nk, d, seed=90 + skip, causal=causal, n_splits=n_splits)
    q, k, v = workloads.generate(w, device="cuda")
    assert fa.device_status() == fa.FA_OK  # clean start
    fa.fwd(q, k, v, w.scale, causal, n_splits, timeout_ns=20_000_000, test_skip_kv_load=skip)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_ERR_DEVICE_TIMEOUT
    assert fa.device_status() == fa.FA_OK  # reading clears the status word
    # the context is still usable and correct
    o, lse = fa.fwd(q, k, v, w.scale, causal, n_splits)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    P.compare(q, k, v, o, lse, w.scale, causal).check("after timeout")
