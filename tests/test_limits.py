"""The largest head count the C ABI accepts: B*H = 65535 (one grid dimension
per (b, h)), through the forward, the split forward, the local mask and the
backward, each checked against the oracle on the first, the last and a middle
head.  Short rows (Nk = 130: two K/V tiles, the second ragged) keep the
tensors near 1 GB each."""
import pytest
import torch

import online_softmax_sm_gb300 as fa
from online_softmax_sm_gb300 import workloads
from tests import _parity as P

pytestmark = pytest.mark.gpu

B, H = 5, 13107  # B * H = 65535
HEADS = [(0, 0), (2, 6553), (4, 13106)]


@pytest.fixture(scope="module")
def qkv():
    w = workloads.custom(B, H, 130, 130, 64, seed=31, q_mult=2.0)
    q, k, v = workloads.generate(w, device="cuda")
    return w, q, k, v


@pytest.mark.parametrize("n_splits", [1, 2])
def test_forward_at_the_head_limit(qkv, n_splits):
    w, q, k, v = qkv
    o, lse = fa.fwd(q, k, v, w.scale, False, n_splits)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    P.compare(q, k, v, o, lse, w.scale, False, heads=HEADS).check(f"B*H = 65535, {n_splits} split(s)")


def test_local_and_causal_at_the_head_limit(qkv):
    w, q, k, v = qkv
    o, lse = fa.fwd_local(q, k, v, 40, 0, w.scale)
    torch.cuda.synchronize()
    P.compare(q, k, v, o, lse, w.scale, False, heads=HEADS, window=(40, 0)).check("B*H = 65535, window")
    o, lse = fa.fwd(q, k, v, w.scale, True)
    torch.cuda.synchronize()
    P.compare(q, k, v, o, lse, w.scale, True, heads=HEADS).check("B*H = 65535, causal")


def test_backward_at_the_head_limit(qkv):
    from tests.test_bwd import _check_head

    w, q, k, v = qkv
    g = torch.Generator(device="cuda")
    g.manual_seed(32)
    do = torch.randn(q.shape, generator=g, device="cuda").to(torch.bfloat16)
    o, lse = fa.fwd(q, k, v, w.scale, True)
    dq, dk, dv = fa.bwd(q, k, v, o, lse, do, w.scale, causal=True)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    for b, h in HEADS:
        f = lambda t: t[b, h].detach().cpu().double().numpy()
        _check_head(f(q), f(k), f(v), f(o), f(do), f(dq), f(dk), f(dv), w.scale, (-1, 0),
                    f"bwd B*H = 65535 head ({b}, {h})")
