"""Attention backward (fa_bwd / fa_bwd_local) against the oracle's gradients.

The kernels take O and LSE from the library's own forward (as a training step
would) and round P^T and dS to bf16 for their MMAs.  Bound per element, from
that arithmetic (u = 2^-9, the bf16 unit roundoff; sums over the visible
pairs, taken from the oracle's exact quantities):
  dV_jc:  2u sum_i P_ij |dO_ic|
  dK_jc:  scale 2u (sum_i |dS_ij| |q_ic| + sum_i P_ij E_i |q_ic|)
  dQ_ic:  scale 2u (sum_j |dS_ij| |k_jc| + E_i sum_j P_ij |k_jc|)
where E_i = sum_c |dO_ic| |O_ic| bounds the error of D_i = <dO_i, O_i> from the
bf16 O.  The factor 2 covers the fp32 exponential, the fp32 accumulations and
the forward's own error in LSE; bf16 results may also differ by half a bf16 ulp
of the reference, and 1e-6 of the largest reference value covers sums that
cancel to about zero.
"""
import numpy as np
import pytest
import torch

import oracle
import online_softmax_sm_gb300 as fa
from online_softmax_sm_gb300 import workloads
from tests import _parity as P

pytestmark = pytest.mark.gpu

U = 2.0 ** -9


def _masks(nq, nk, window, r0=0, r1=None):
    """Visible (query, key) pairs of query rows [r0, r1) (all by default)."""
    wl, wr = window
    r1 = nq if r1 is None else r1
    i = np.arange(r0, r1)[:, None] + (nk - nq)
    j = np.arange(nk)[None, :]
    vis = np.ones((r1 - r0, nk), dtype=bool)
    if wl >= 0:
        vis &= j >= i - wl
    if wr >= 0:
        vis &= j <= i + wr
    return vis


def _check_head(q, k, v, o, do, dq, dk, dv, scale, window, what, block=1024):
    """One head, all elements; q, k, v, o, do, dq, dk, dv: CPU float64 numpy.
    The bounds are summed over blocks of query rows, so the nq x nk
    matrices never exist whole."""
    ref = oracle.attention_bwd(q, k, v, do, scale, window=window)
    nq, nk = q.shape[0], k.shape[0]
    e = np.sum(np.abs(do) * np.abs(o), axis=1)
    bounds = {"dv": np.zeros_like(v), "dk": np.zeros_like(k), "dq": np.zeros_like(q)}
    for r0 in range(0, nq, block):
        r = slice(r0, min(nq, r0 + block))
        vis = _masks(nq, nk, window, r.start, r.stop)
        lse = ref["lse"][r, None]
        live = np.isfinite(lse)
        s = scale * (q[r] @ k.T)
        pm = np.where(vis & live, np.exp(np.where(vis & live, s - np.where(live, lse, 0.0), -np.inf)), 0.0)
        ds = pm * (do[r] @ v.T - ref["dd"][r, None])
        bounds["dv"] += 2 * U * (pm.T @ np.abs(do[r]))
        bounds["dk"] += scale * 2 * U * (np.abs(ds).T @ np.abs(q[r]) + (pm * e[r, None]).T @ np.abs(q[r]))
        bounds["dq"][r] = scale * 2 * U * (np.abs(ds) @ np.abs(k) + e[r, None] * (pm @ np.abs(k)))
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        r = ref[name]
        tol = bounds[name] + P.half_ulp_bf16(r) + 1e-6 * np.abs(r).max(initial=0.0)
        err = np.abs(got - r)
        bad = err > tol
        assert not bad.any(), (f"{what} {name}: {bad.sum()} of {bad.size} out of bound, worst excess "
                               f"{(err - tol).max():.3e}, max|d|={err.max():.3e}, max|ref|={np.abs(r).max():.3e}")


def _run(B, H, Nq, Nk, d, window, seed, q_mult=1.0):
    w = workloads.custom(B, H, Nq, Nk, d, seed=seed, q_mult=q_mult)
    q, k, v = workloads.generate(w, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(seed + 1000)
    do = torch.randn(q.shape, generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    wl, wr = window
    if window == (-1, -1) or window == (-1, 0):
        o, lse = fa.fwd(q, k, v, w.scale, window == (-1, 0))
        dq, dk, dv = fa.bwd(q, k, v, o, lse, do, w.scale, causal=(window == (-1, 0)))
    else:
        o, lse = fa.fwd_local(q, k, v, wl, wr, w.scale)
        dq, dk, dv = fa.bwd(q, k, v, o, lse, do, w.scale, window=window)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    return w, q, k, v, o, lse, do, dq, dk, dv


def _np(t):
    return t.detach().cpu().double().numpy()


# B, H, Nq, Nk, d, window
CASES = [
    (1, 2, 256, 256, 128, (-1, -1)),
    (1, 2, 256, 256, 128, (-1, 0)),
    (1, 1, 200, 333, 64, (-1, -1)),
    (2, 1, 300, 300, 128, (-1, 0)),
    (1, 2, 384, 129, 64, (-1, 0)),     # Nq > Nk: rows with no key; a one-key tail tile
    (1, 1, 130, 700, 128, (-1, 0)),    # decode-like, ragged
    (1, 1, 512, 512, 128, (100, 0)),   # sliding window
    (1, 2, 257, 400, 64, (30, 40)),    # two-sided window, ragged
    # d = 64 with more 128-row tiles than any ring has slots (four each), so
    # every Q, dO, K and V slot is reused
    (1, 1, 700, 650, 64, (-1, -1)),
    (1, 1, 640, 767, 64, (-1, 0)),
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,window", CASES,
                         ids=[f"b{c[0]}h{c[1]}nq{c[2]}nk{c[3]}d{c[4]}w{c[5][0]}_{c[5][1]}" for c in CASES])
def test_bwd_all_elements(B, H, Nq, Nk, d, window):
    w, q, k, v, o, _, do, dq, dk, dv = _run(B, H, Nq, Nk, d, window, seed=Nq + Nk + d)
    for b in range(B):
        for h in range(H):
            _check_head(_np(q[b, h]), _np(k[b, h]), _np(v[b, h]), _np(o[b, h]), _np(do[b, h]),
                        _np(dq[b, h]), _np(dk[b, h]), _np(dv[b, h]), w.scale, window,
                        f"{w.name} w={window} (b={b},h={h})")


def test_bwd_repeats_bit_exact():
    """No atomics: two calls on the same inputs give the same bits."""
    w, q, k, v, o, lse, do, dq, dk, dv = _run(1, 4, 640, 640, 128, (-1, 0), seed=5)
    dq2, dk2, dv2 = fa.bwd(q, k, v, o, lse, do, w.scale, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(dq, dq2) and torch.equal(dk, dk2) and torch.equal(dv, dv2)


def test_bwd_full_size_head():
    """The non-causal d = 128, N = 4096 shape (Q x4): one head of the full
    call checked element by element."""
    w = workloads.C3
    q, k, v = workloads.generate(w, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(77)
    do = torch.randn(q.shape, generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    o, lse = fa.fwd(q, k, v, w.scale, False)
    dq, dk, dv = fa.bwd(q, k, v, o, lse, do, w.scale, causal=False)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    b, h = 1, 17
    _check_head(_np(q[b, h]), _np(k[b, h]), _np(v[b, h]), _np(o[b, h]), _np(do[b, h]), _np(dq[b, h]),
                _np(dk[b, h]), _np(dv[b, h]), w.scale, (-1, -1), w.name)


@pytest.mark.parametrize("name", ["c4", "local"])
def test_bwd_full_size_head_causal_and_window(name):
    """The causal N = 16384 shape and the 4096-key window on it, as the
    benchmark runs them: one head of the full call, element by element."""
    w = workloads.C4 if name == "c4" else workloads.LOCAL
    window = w.window if w.window is not None else (-1, 0)
    q, k, v = workloads.generate(w, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(78)
    do = torch.randn(q.shape, generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    if w.window is not None:
        o, lse = fa.fwd_local(q, k, v, window[0], window[1], w.scale)
    else:
        o, lse = fa.fwd(q, k, v, w.scale, True)
    dq, dk, dv = fa.bwd(q, k, v, o, lse, do, w.scale, causal=w.causal, window=w.window)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    b, h = 0, 21
    _check_head(_np(q[b, h]), _np(k[b, h]), _np(v[b, h]), _np(o[b, h]), _np(do[b, h]), _np(dq[b, h]),
                _np(dk[b, h]), _np(dv[b, h]), w.scale, window, w.name)


@pytest.mark.parametrize("d", [64, 128])
def test_bwd_bad_arguments(d):
    w = workloads.custom(1, 1, 128, 128, d, seed=1)
    q, k, v = workloads.generate(w, device="cuda")
    lse = torch.zeros((1, 1, 128), device="cuda")
    with pytest.raises(fa.FAError):
        fa.bwd(q, k, v, q, lse, q, 0.0)  # scale must be > 0
    with pytest.raises(fa.FAError):
        fa.bwd(q, k, v, q, lse, q, 0.1, window=(-2, 0))
