"""Seeded synthetic inputs for the attention forward.

This module holds none of the method's arithmetic: it only draws Q, K and V.
Both the GPU path's tests/benchmark and the fp64 oracle consume what it
produces (the oracle gets the very same bf16 values, upcast exactly).

Recipe (per workload): a torch.Generator on the target device seeded with
`seed`; fp32 N(0, 1) draws for Q, then K, then V, in that order; optional
structure (Q multiplied by `q_mult`; K row j multiplied by 1 + j/Nk when
`k_ramp`); then a round-to-nearest cast to bf16.  Layout [B, H, N, d],
contiguous.  Draws on CPU and on CUDA differ for the same seed; each run is
self-consistent because both sides read the same tensors.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    causal: bool = False
    n_splits: int = 1
    bc: int = 0            # K/V tile override (0: library default)
    q_mult: float = 1.0    # Q scaled by this (logit spread)
    k_ramp: bool = False   # K row j scaled by 1 + j/Nk (running max grows across tiles)
    seed: int = 0
    # Local mask (window_left, window_right): key j visible to query i iff
    # i + (Nk - Nq) - window_left <= j <= i + (Nk - Nq) + window_right, -1 = open
    # side.  None: the plain or causal mask of `causal`.
    window: tuple[int, int] | None = None

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def visible_pairs(self) -> int:
        """Number of (query, key) pairs the mask leaves visible, per head."""
        if self.window is None:
            return self.Nq * self.Nk
        wl, wr = self.window
        i = np.arange(self.Nq, dtype=np.int64) + (self.Nk - self.Nq)
        lo = np.zeros_like(i) if wl < 0 else np.maximum(i - wl, 0)
        hi = np.full_like(i, self.Nk - 1) if wr < 0 else np.minimum(i + wr, self.Nk - 1)
        return int(np.maximum(hi - lo + 1, 0).sum())

    @property
    def flops(self) -> float:
        """Algorithmic FLOPs: 4*d per visible (query, key) pair; for causal
        without a window, the usual 4*B*H*Nq*Nk*d / 2."""
        if self.window is not None:
            return 4.0 * self.B * self.H * self.d * self.visible_pairs()
        f = 4.0 * self.B * self.H * self.Nq * self.Nk * self.d
        return f / 2 if self.causal else f

    @property
    def io_bytes(self) -> int:
        """Algorithmic HBM bytes: read Q, K, V (bf16) once; write O (bf16) and LSE (fp32)."""
        q = self.B * self.H * self.Nq * self.d * 2
        kv = 2 * self.B * self.H * self.Nk * self.d * 2
        o = self.B * self.H * self.Nq * self.d * 2
        lse = self.B * self.H * self.Nq * 4
        return q + kv + o + lse

    def describe(self) -> dict:
        d = dataclasses.asdict(self)
        d["scale"] = self.scale
        return d


# The five workloads the path is specified on.
C1 = Workload("noncausal_b1h1n256d64_bc64", 1, 1, 256, 256, 64, bc=64, seed=0)
C2 = Workload("noncausal_b4h16n1024d64", 4, 16, 1024, 1024, 64, seed=1)
C3 = Workload("noncausal_b2h32n4096d128_q4", 2, 32, 4096, 4096, 128, q_mult=4.0, seed=2)
C4 = Workload("causal_b1h32n16384d128_kramp", 1, 32, 16384, 16384, 128, causal=True, k_ramp=True, seed=3)
# Companion call to C4: 256 fewer keys, so under bottom-right causal alignment
# query rows 0..255 see no key at all (the fully masked rows).
C4_MASKED = Workload("causal_b1h32nq16384nk16128d128_kramp", 1, 32, 16384, 16384 - 256, 128,
                     causal=True, k_ramp=True, seed=3)
C5 = Workload("splitkv_b16h32nq128nk32768d128_s16", 16, 32, 128, 32768, 128, n_splits=16, seed=4)
# Local mask: causal sliding window of 4096 keys (the query's own key and the
# 4095 before it) over a 16K sequence.
LOCAL = Workload("local_b1h32n16384d128_w4096", 1, 32, 16384, 16384, 128, window=(4095, 0),
                 k_ramp=True, seed=5)

WORKLOADS = {w.name: w for w in (C1, C2, C3, C4, C4_MASKED, C5, LOCAL)}


@dataclasses.dataclass(frozen=True)
class SoftmaxWorkload:
    """Rows of logits for the standalone softmax: fp32 N(0, sigma^2) draws,
    cast to `dtype` ("f32" or "bf16"), [rows, cols] contiguous."""
    name: str
    rows: int
    cols: int
    dtype: str = "f32"
    sigma: float = 4.0
    seed: int = 0

    @property
    def elt(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def io_bytes(self) -> int:
        """Algorithmic HBM bytes: read x once, write y once and one fp32 LSE per row."""
        return 2 * self.rows * self.cols * self.elt + 4 * self.rows

    def describe(self) -> dict:
        return dataclasses.asdict(self)


# Attention-score rows (B*H*N rows of N scores: 32 heads x 1024 queries of a
# 4096-token context) and a language-model head's logits over a 128K
# vocabulary; the long-row case exceeds what a CTA cluster keeps on chip.
SOFTMAX_F32 = SoftmaxWorkload("softmax_f32_r32768c4096", 32768, 4096, "f32", seed=7)
SOFTMAX_BF16_VOCAB = SoftmaxWorkload("softmax_bf16_r4096c131072", 4096, 131072, "bf16", seed=8)
SOFTMAX_F32_LONG = SoftmaxWorkload("softmax_f32_r256c1048576", 256, 1 << 20, "f32", seed=9)
SOFTMAX_WORKLOADS = {w.name: w for w in (SOFTMAX_F32, SOFTMAX_BF16_VOCAB, SOFTMAX_F32_LONG)}


def generate_logits(w: SoftmaxWorkload, device="cpu") -> torch.Tensor:
    """Draw x for softmax workload `w` on `device`."""
    g = torch.Generator(device=device)
    g.manual_seed(w.seed)
    x = torch.randn((w.rows, w.cols), generator=g, device=device, dtype=torch.float32)
    x.mul_(w.sigma)
    return x if w.dtype == "f32" else x.to(torch.bfloat16)


def generate(w: Workload, device="cpu", dtype=torch.bfloat16):
    """Draw (q, k, v) for workload `w` on `device` ([B,H,N,d], contiguous)."""
    g = torch.Generator(device=device)
    g.manual_seed(w.seed)
    shape_q = (w.B, w.H, w.Nq, w.d)
    shape_kv = (w.B, w.H, w.Nk, w.d)
    q = torch.randn(shape_q, generator=g, device=device, dtype=torch.float32)
    if w.q_mult != 1.0:
        q.mul_(w.q_mult)
    q = q.to(dtype)
    k = torch.randn(shape_kv, generator=g, device=device, dtype=torch.float32)
    if w.k_ramp:
        ramp = 1.0 + torch.arange(w.Nk, device=device, dtype=torch.float32) / w.Nk
        k.mul_(ramp.view(1, 1, -1, 1))
    k = k.to(dtype)
    v = torch.randn(shape_kv, generator=g, device=device, dtype=torch.float32).to(dtype)
    return q, k, v


def custom(B, H, Nq, Nk, d, seed=0, causal=False, n_splits=1, bc=0, q_mult=1.0, k_ramp=False,
           name=None, window=None) -> Workload:
    return Workload(name or f"b{B}h{H}nq{Nq}nk{Nk}d{d}", B, H, Nq, Nk, d, causal=causal,
                    n_splits=n_splits, bc=bc, q_mult=q_mult, k_ramp=k_ramp, seed=seed,
                    window=None if window is None else tuple(window))
