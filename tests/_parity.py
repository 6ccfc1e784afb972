"""Shared helpers for the GPU parity tests: run the CUDA path, run the fp64
oracle on the same bf16 inputs, compare element by element.

Tolerance (bf16 inputs, fp32 accumulation): max |dO| <= 1e-2,
mean |dO| <= 1e-3, max |dLSE| <= 1e-3.  Rows the oracle marks fully masked
(LSE = -inf) must come back with O exactly 0 and LSE exactly -inf.

The bound is applied to the kernel's computed (fp32) O, which the same kernel
emits through its partial-output epilogue (fa_fwd_partial with one split).
The bf16 O of fa_fwd must then be exactly that fp32 value rounded to nearest
even, and is compared with the oracle at the bound plus half a bf16 ulp of the
reference value: for |O| >= 4 the bf16 grid spacing (2^-5) alone exceeds 1e-2.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import online_softmax_sm_gb300 as fa
from online_softmax_sm_gb300 import workloads

MAX_ABS_O = 1e-2
MEAN_ABS_O = 1e-3
MAX_ABS_LSE = 1e-3


class Diff:
    def __init__(self):
        self.max_o = 0.0
        self.sum_o = 0.0
        self.n_o = 0
        self.max_lse = 0.0
        self.rows = 0
        self.masked_rows = 0

    def add(self, o_gpu: np.ndarray, lse_gpu: np.ndarray, o_ref: np.ndarray, lse_ref: np.ndarray,
            bf16_output: bool = False):
        masked = np.isneginf(lse_ref)
        if masked.any():
            assert np.all(o_gpu[masked] == 0.0), "masked rows must give O = 0 exactly"
            assert np.all(np.isneginf(lse_gpu[masked])), "masked rows must give LSE = -inf"
        keep = ~masked
        assert np.all(np.isfinite(o_gpu)), "non-finite O"
        assert np.all(np.isfinite(lse_gpu[keep])), "non-finite LSE on a visible row"
        d = np.abs(o_gpu - o_ref)
        self.max_o_raw = max(getattr(self, "max_o_raw", 0.0), float(d.max(initial=0.0)))
        # bf16 output: discount the storage rounding (half an ulp of the reference)
        dm = np.maximum(d - half_ulp_bf16(o_ref), 0.0) if bf16_output else d
        self.max_o = max(self.max_o, float(dm.max(initial=0.0)))
        self.sum_o += float(d.sum())
        self.n_o += d.size
        if keep.any():
            self.max_lse = max(self.max_lse, float(np.abs(lse_gpu[keep] - lse_ref[keep]).max()))
        self.rows += o_gpu.shape[0]
        self.masked_rows += int(masked.sum())

    @property
    def mean_o(self):
        return self.sum_o / max(self.n_o, 1)

    def check(self, what=""):
        msg = (f"{what}: rows={self.rows} masked={self.masked_rows} max|dO|={self.max_o:.3e} "
               f"(raw {getattr(self, 'max_o_raw', self.max_o):.3e}) "
               f"mean|dO|={self.mean_o:.3e} max|dLSE|={self.max_lse:.3e}")
        assert self.max_o <= MAX_ABS_O, msg
        assert self.mean_o <= MEAN_ABS_O, msg
        assert self.max_lse <= MAX_ABS_LSE, msg
        return msg


def half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Half the spacing of the bf16 grid at |x| (8 significand bits)."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, np.exp2(e - 8), 0.0)


def compare_many(q, k, v, outs, scale, causal, heads=None, rows=None, threads=None,
                 window=None) -> list[Diff]:
    """outs: list of (o, lse) pairs for the same q, k, v; one oracle run per
    head serves all of them.  q/k/v/o: [B,H,N,d] (any device), lse [B,H,Nq];
    heads: list of (b,h).  A bf16 `o` is compared with the half-ulp storage
    allowance, fp32 `o` without.  window=(wl, wr): the oracle's local mask
    instead of `causal`."""
    diffs = [Diff() for _ in outs]
    B, H = q.shape[0], q.shape[1]
    every = heads is None
    heads = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    # every head: one copy of each tensor to the host; a few heads: per head
    host = (lambda t: t.cpu()) if every else (lambda t: t)
    qc, kc, vc = host(q), host(k), host(v)
    outs_c = [(host(o), host(lse), o.dtype == torch.bfloat16) for o, lse in outs]
    for (b, h) in heads:
        qh, kh, vh = qc[b, h].cpu(), kc[b, h].cpu(), vc[b, h].cpu()
        if window is None:
            o_ref, lse_ref = oracle.attention(qh, kh, vh, scale, causal, rows=rows, threads=threads)
        else:
            o_ref, lse_ref = oracle.attention_window(qh, kh, vh, scale, window[0], window[1], rows=rows,
                                                     threads=threads)
        for diff, (o, lse, bf16_out) in zip(diffs, outs_c):
            og = o[b, h].cpu().double().numpy()
            lg = lse[b, h].cpu().double().numpy()
            if rows is not None:
                og, lg = og[rows], lg[rows]
            diff.add(og, lg, o_ref, lse_ref, bf16_output=bf16_out)
    return diffs


def compare(q, k, v, o, lse, scale, causal, heads=None, rows=None, diff: Diff | None = None,
            threads=None, window=None) -> Diff:
    """One output pair against the oracle (see compare_many)."""
    d = compare_many(q, k, v, [(o, lse)], scale, causal, heads=heads, rows=rows, threads=threads,
                     window=window)[0]
    if diff is None:
        return d
    diff.max_o = max(diff.max_o, d.max_o)
    diff.max_o_raw = max(getattr(diff, "max_o_raw", 0.0), getattr(d, "max_o_raw", 0.0))
    diff.sum_o += d.sum_o
    diff.n_o += d.n_o
    diff.max_lse = max(diff.max_lse, d.max_lse)
    diff.rows += d.rows
    diff.masked_rows += d.masked_rows
    return diff


def run_workload(w: workloads.Workload, heads=None, rows=None, n_splits=None, bc=None, qt=0):
    """fa_fwd (bf16 O) and the same kernel's fp32 result (fa_fwd_partial, one
    split), both against the oracle; the bf16 O must be the fp32 result
    rounded to nearest even, bit for bit, when no merge is involved."""
    q, k, v = workloads.generate(w, device="cuda")
    ns = w.n_splits if n_splits is None else n_splits
    bcv = w.bc if bc is None else bc
    o, lse = fa.fwd(q, k, v, w.scale, w.causal, ns, bc=bcv, q_tiles_per_cta=qt)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    if not (bcv in (0, 128) and qt == 0):
        d_bf16 = compare(q, k, v, o, lse, w.scale, w.causal, heads=heads, rows=rows)
        d_bf16.check(w.name + " (bf16 O)")
        return d_bf16
    m_p, l_p, o_p = fa.fwd_partial(q, k, v, 1, w.scale, w.causal)
    torch.cuda.synchronize()
    lse32 = torch.where(l_p[0] > 0, m_p[0].double() + torch.log(l_p[0].double()),
                        torch.full_like(l_p[0], float("-inf"), dtype=torch.float64))
    d_bf16, d32 = compare_many(q, k, v, [(o, lse), (o_p[0], lse32)], w.scale, w.causal, heads=heads,
                               rows=rows)
    d_bf16.check(w.name + " (bf16 O)")
    d32.check(w.name + " (fp32 O)")
    if ns == 1:
        assert torch.equal(o, o_p[0].to(torch.bfloat16)), "bf16 O is not RNE of the fp32 result"
        fin = torch.isfinite(lse)
        assert torch.equal(fin, torch.isfinite(lse32))
        assert (lse[fin].double() - lse32[fin]).abs().max().item() <= 1e-5
    return d32


def sample_rows(nq: int, tile: int = 128, extra: int = 64, seed: int = 0) -> list[int]:
    """Every tile's first and last row, the last row overall, plus seeded extras."""
    rng = np.random.default_rng(seed)
    rows = set()
    for t0 in range(0, nq, tile):
        rows.add(t0)
        rows.add(min(t0 + tile, nq) - 1)
    rows.update(rng.integers(0, nq, size=extra).tolist())
    return sorted(rows)
