"""fa_fwd_host (host buffers, copies included) against fa_fwd on the device.

fa_fwd_host runs the same kernel on groups of consecutive (b, h) heads, so its
O and LSE must equal fa_fwd's bit for bit for any grouping; fa_fwd itself is
held to the oracle by the parity tests.  Cases cover groupings that divide
B*H, that do not, one group per head, more groups than heads, causal masks,
ragged lengths, page-locked and pageable host memory, and a second call that
reuses (and a larger one that grows) the library's device buffer.
"""
import pytest
import torch

import online_softmax_sm_gb300 as fa
from online_softmax_sm_gb300 import workloads

pytestmark = pytest.mark.gpu


def _case(B, H, Nq, Nk, d, causal, seed, n_chunks, pinned=True):
    w = workloads.custom(B, H, Nq, Nk, d, seed=seed, q_mult=2.0, causal=causal)
    q, k, v = workloads.generate(w, device="cuda")
    o_ref, lse_ref = fa.fwd(q, k, v, w.scale, causal)
    torch.cuda.synchronize()
    hq, hk, hv = (t.cpu() for t in (q, k, v))
    if pinned:
        hq, hk, hv = (t.pin_memory() for t in (hq, hk, hv))
    o, lse = fa.fwd_host(hq, hk, hv, w.scale, causal, n_chunks=n_chunks)
    assert o.device.type == "cpu" and lse.device.type == "cpu"
    assert torch.equal(o, o_ref.cpu()), f"O differs ({B},{H},{Nq},{Nk},{d}, chunks={n_chunks})"
    assert torch.equal(lse, lse_ref.cpu()), f"LSE differs ({B},{H},{Nq},{Nk},{d}, chunks={n_chunks})"


# B, H, Nq, Nk, d, causal, n_chunks
CASES = [
    (2, 4, 512, 512, 128, False, 0),     # default grouping: 8 groups of one head
    (2, 4, 512, 512, 128, False, 3),     # 3 groups of 3, 3, 2 heads
    (1, 6, 300, 700, 64, False, 4),      # ragged lengths, d = 64
    (1, 4, 1024, 1024, 128, True, 2),    # causal
    (1, 3, 200, 200, 128, True, 10),     # more groups than heads (clamped)
    (1, 1, 1, 1, 64, False, 0),          # one row, one key
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,n_chunks", CASES,
                         ids=[f"b{c[0]}h{c[1]}nq{c[2]}nk{c[3]}d{c[4]}{'c' if c[5] else ''}g{c[6]}" for c in CASES])
def test_fwd_host_matches_device_call(B, H, Nq, Nk, d, causal, n_chunks):
    _case(B, H, Nq, Nk, d, causal, seed=Nq + Nk + H, n_chunks=n_chunks)


def test_fwd_host_pageable_memory():
    _case(1, 4, 384, 384, 128, False, seed=3, n_chunks=2, pinned=False)


def test_fwd_host_buffer_reuse_and_growth():
    _case(1, 2, 256, 256, 64, False, seed=1, n_chunks=2)
    _case(1, 2, 256, 256, 64, False, seed=2, n_chunks=2)     # same size: buffer reused
    _case(2, 8, 1024, 2048, 128, False, seed=3, n_chunks=0)  # larger: buffer grows


def test_fwd_host_rejects_bad_arguments():
    q = torch.zeros((1, 1, 128, 128), dtype=torch.bfloat16)
    with pytest.raises(fa.FAError):
        fa.fwd_host(q, q, q, 0.0)           # scale must be > 0
    with pytest.raises(ValueError):
        fa.fwd_host(q.cuda(), q, q)         # device tensors belong to fa.fwd
    rc = fa.lib().fa_fwd_host(None, q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(),
                              1, 1, 128, 128, 128, 0.1, 0, 0)
    assert rc == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("window,n_chunks", [((64, 0), 3), ((200, 50), 0), ((-1, 0), 2)])
def test_fwd_local_host_matches_device_call(window, n_chunks):
    """fa_fwd_local_host against fa_fwd_local: the same kernel per head group."""
    w = workloads.custom(1, 4, 300, 500, 128, seed=7, q_mult=2.0)
    q, k, v = workloads.generate(w, device="cuda")
    o_ref, lse_ref = fa.fwd_local(q, k, v, window[0], window[1], w.scale)
    torch.cuda.synchronize()
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    o, lse = fa.fwd_host(hq, hk, hv, w.scale, n_chunks=n_chunks, window=window)
    assert torch.equal(o, o_ref.cpu()) and torch.equal(lse, lse_ref.cpu())


@pytest.mark.parametrize("causal,n_chunks", [(False, 3), (True, 0)])
def test_fwd_fp8_host_matches_device_call(causal, n_chunks):
    """fa_fwd_fp8_host against fa_fwd_fp8 (one-byte inputs, bf16 O)."""
    w = workloads.custom(2, 3, 384, 300, 128, seed=8)
    q8, k8, v8 = (t.to(torch.float8_e4m3fn) for t in workloads.generate(w, device="cuda"))
    o_ref, lse_ref = fa.fwd_fp8(q8, k8, v8, w.scale, 0.5, 1.0, 2.0, causal)
    torch.cuda.synchronize()
    hq, hk, hv = (t.cpu().pin_memory() for t in (q8, k8, v8))
    o, lse = fa.fwd_fp8_host(hq, hk, hv, w.scale, 0.5, 1.0, 2.0, causal, n_chunks=n_chunks)
    assert torch.equal(o, o_ref.cpu()) and torch.equal(lse, lse_ref.cpu())


@pytest.mark.parametrize("window,n_chunks", [(None, 3), ((-1, 0), 0), ((100, 0), 4)])
def test_bwd_host_matches_device_call(window, n_chunks):
    """fa_bwd_host / fa_bwd_local_host against fa_bwd on the device (no atomics,
    heads independent: equal bit for bit for any grouping)."""
    w = workloads.custom(1, 5, 300, 260, 128, seed=9)
    q, k, v = workloads.generate(w, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(10)
    do = torch.randn(q.shape, generator=g, device="cuda").to(torch.bfloat16)
    if window is None:
        o, lse = fa.fwd(q, k, v, w.scale)
    else:
        o, lse = fa.fwd_local(q, k, v, window[0], window[1], w.scale)
    ref = fa.bwd(q, k, v, o, lse, do, w.scale, window=window)
    torch.cuda.synchronize()
    h = [t.cpu().pin_memory() for t in (q, k, v, o, lse, do)]
    got = fa.bwd_host(*h, w.scale, window=window, n_chunks=n_chunks)
    for a, b in zip(got, ref):
        assert torch.equal(a, b.cpu())
