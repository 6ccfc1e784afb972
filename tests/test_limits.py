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


def test_keys_past_4_gib_in_one_head():
    """One head with Nk = 2^25 keys at d = 64: K and V hold 4 GiB each, so
    every byte offset past the first 2^32 must be formed in 64 bits.  The
    reference for sampled rows comes from the oracle over key chunks of 2^22,
    combined with the oracle's merge rule (the rows see every key)."""
    import numpy as np

    import oracle

    Nq, Nk, d = 128, 1 << 25, 64
    w = workloads.custom(1, 1, Nq, Nk, d, seed=33)
    q, k, v = workloads.generate(w, device="cuda")
    rows = [0, 1, 31, 64, 100, 127]
    qh = q[0, 0].cpu().double().numpy()
    parts_o, parts_lse = [], []
    chunk = 1 << 22
    for c0 in range(0, Nk, chunk):
        kc = k[0, 0, c0:c0 + chunk].cpu().double().numpy()
        vc = v[0, 0, c0:c0 + chunk].cpu().double().numpy()
        o_c, lse_c = oracle.attention(qh, kc, vc, w.scale, False, rows=rows)
        parts_o.append(o_c)
        parts_lse.append(lse_c)
        del kc, vc
    o_ref = np.empty((len(rows), d))
    lse_ref = np.empty(len(rows))
    for r in range(len(rows)):
        # a chunk's (O, LSE) is the partial (m = LSE, l = 1, O) of the merge rule
        m = np.array([p[r] for p in parts_lse])
        _, _, o_r, lse_r = oracle.merge(m, np.ones_like(m), np.stack([p[r] for p in parts_o]))
        o_ref[r], lse_ref[r] = o_r, lse_r
    for n_splits in (1, 296):
        o, lse = fa.fwd(q, k, v, w.scale, False, n_splits)
        torch.cuda.synchronize()
        assert fa.device_status() == fa.FA_OK
        diff = P.Diff()
        diff.add(o[0, 0, rows].float().cpu().double().numpy(), lse[0, 0, rows].cpu().double().numpy(),
                 o_ref, lse_ref, bf16_output=True)
        print(diff.check(f"Nk = 2^25, d = 64, {n_splits} split(s)"))


def test_softmax_past_2_31_elements():
    """2049 rows of 2^20 bf16 logits: 2^31 + 2^20 elements (4.3 GB); rows at
    both ends and in the middle against the oracle's two-pass normaliser."""
    from tests.test_softmax import _check

    sw = workloads.SoftmaxWorkload("limit", 2049, 1 << 20, "bf16", seed=34)
    x = workloads.generate_logits(sw, device="cuda")
    y, lse = fa.softmax_rows(x)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    rows = torch.tensor([0, 1, 1024, 2047, 2048], device="cuda")
    # only the sampled rows go to the host (the whole matrix in fp64 would be 17 GB)
    _check(x[rows], y[rows], lse[rows], what="2049 x 2^20 bf16")
