"""Local (sliding-window) mask: fa_fwd_local against the oracle's windowed
attention, every row, plus the identities that tie it to fa_fwd.

Mask ("Online Softmax 算法详解", section 3.2, names causal and local masks):
key j is visible to query i iff i + off - wl <= j <= i + off + wr with
off = Nk - Nq and -1 leaving a side open.  The kernel skips K/V tiles that lie
wholly outside a query tile's window, so the cases put windows on tile
boundaries, inside one tile, across several tiles, far from the first key,
and make some query tiles (or rows) see no key at all.
"""
import pytest
import torch

import online_softmax_sm_gb300 as fa
from online_softmax_sm_gb300 import workloads
from tests import _parity as P

pytestmark = pytest.mark.gpu

# B, H, Nq, Nk, d, window_left, window_right, n_splits
CASES = [
    (1, 2, 512, 512, 128, 127, 0, 1),      # causal sliding window of 128 keys
    (1, 2, 700, 900, 64, 200, 50, 1),      # two-sided, Nq != Nk, ragged tails
    (2, 1, 300, 300, 128, 0, 0, 1),        # the diagonal only: one key per row
    (1, 2, 640, 640, 128, 64, 64, 3),      # symmetric, split-KV
    (1, 1, 1000, 1000, 128, -1, 300, 1),   # left side open, 300 keys of look-ahead
    (1, 1, 600, 600, 64, 257, -1, 1),      # right side open
    (1, 2, 400, 200, 128, 50, 0, 1),       # off < 0: rows 0..199 see no key
    (1, 2, 256, 100, 64, 20, 0, 1),        # first query tile sees nothing, second does
    (1, 1, 256, 4096, 128, 1000, 0, 4),    # splits wholly outside the window
    (1, 1, 200, 1500, 128, 10, 10, 1),     # window far from key 0
    (1, 2, 100, 800, 128, 30, 5, 1),       # one query tile per CTA
    (1, 1, 384, 1024, 128, 130, 129, 2),   # windows straddling tile edges, splits
]


def _run(B, H, Nq, Nk, d, wl, wr, ns, seed, q_mult=2.0):
    w = workloads.custom(B, H, Nq, Nk, d, seed=seed, q_mult=q_mult, window=(wl, wr), n_splits=ns)
    q, k, v = workloads.generate(w, device="cuda")
    o, lse = fa.fwd_local(q, k, v, wl, wr, w.scale, ns)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    return w, q, k, v, o, lse


@pytest.mark.parametrize("B,H,Nq,Nk,d,wl,wr,ns", CASES,
                         ids=[f"b{c[0]}h{c[1]}nq{c[2]}nk{c[3]}d{c[4]}w{c[5]}_{c[6]}s{c[7]}"
                              for c in CASES])
def test_local_all_rows(B, H, Nq, Nk, d, wl, wr, ns):
    w, q, k, v, o, lse = _run(B, H, Nq, Nk, d, wl, wr, ns, seed=Nq + 3 * Nk + wl)
    diff = P.compare(q, k, v, o, lse, w.scale, False, window=(wl, wr))
    diff.check(w.name + f" window ({wl},{wr})")
    off = Nk - Nq
    want_empty = sum(1 for i in range(Nq)
                     if (wr >= 0 and i + off + wr < 0) or (wl >= 0 and i + off - wl > Nk - 1))
    assert diff.masked_rows == B * H * want_empty


@pytest.mark.parametrize("Nq,Nk,d,ns", [(512, 512, 128, 1), (300, 700, 64, 1), (640, 2000, 128, 3)])
def test_window_bounds_that_reduce_to_fwd_are_bit_exact(Nq, Nk, d, ns):
    """(-1, 0) is fa_fwd's causal mask and (-1, -1) no mask; a left bound
    beyond the key axis changes nothing either.  Same kernel, same tiles:
    the results must be identical bit for bit."""
    w = workloads.custom(1, 2, Nq, Nk, d, seed=5, q_mult=2.0)
    q, k, v = workloads.generate(w, device="cuda")
    for causal, windows in ((True, [(-1, 0), (Nk + Nq, 0)]), (False, [(-1, -1), (Nk + Nq, -1)])):
        o_ref, l_ref = fa.fwd(q, k, v, w.scale, causal, ns)
        for wl, wr in windows:
            o, l = fa.fwd_local(q, k, v, wl, wr, w.scale, ns)
            torch.cuda.synchronize()
            assert torch.equal(o, o_ref), (causal, wl, wr)
            assert torch.equal(l, l_ref), (causal, wl, wr)
    assert fa.device_status() == fa.FA_OK


def test_diagonal_window_returns_v():
    """Window (0, 0) with Nq == Nk: each row sees exactly its own key, so
    softmax is 1 there and O_i = v_i exactly, LSE_i = scale * q_i.k_i."""
    w, q, k, v, o, lse = _run(1, 2, 384, 384, 128, 0, 0, 1, seed=21)
    assert torch.equal(o, v)
    dots = (q.double() * k.double()).sum(-1) * w.scale
    assert (lse.double() - dots).abs().max().item() <= 1e-3


def test_local_workload_sampled():
    """The sliding-window workload (causal window of 4096 keys, 16K tokens,
    32 heads, d = 128) in the launch configuration the benchmark times:
    every tile's first and last row plus seeded extras, on four heads."""
    w = workloads.LOCAL
    q, k, v = workloads.generate(w, device="cuda")
    o, lse = fa.fwd_local(q, k, v, w.window[0], w.window[1], w.scale, w.n_splits)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    rows = P.sample_rows(w.Nq, extra=96, seed=17)
    heads = [(0, 0), (0, 9), (0, 22), (0, 31)]
    P.compare(q, k, v, o, lse, w.scale, False, heads=heads, rows=rows,
              window=w.window).check(w.name)


@pytest.mark.parametrize("wl,wr", [(-2, 0), (0, -5), (2**30 + 1, 0)])
def test_bad_window_is_rejected_before_launch(wl, wr):
    w = workloads.custom(1, 1, 128, 128, 64, seed=1)
    q, k, v = workloads.generate(w, device="cuda")
    o = torch.full_like(q, 7.0)
    with pytest.raises(fa.FAError) as e:
        fa.fwd_local(q, k, v, wl, wr, w.scale, 1, out=o)
    assert e.value.code == fa.FA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.all(o == 7.0)
