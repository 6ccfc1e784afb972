"""FP8 (E4M3) forward with Max_offset = 8 against the oracle's FP8 steps
("Online Softmax 算法详解" section 6), every element.

Where floating point decides a quantised code, both sides should decide in
the same precision; the kernel takes the E4M3 rounding of P' from its fp32
value (ex2.approx of one FFMA), the oracle from fp64.  The two can differ
only where the exact P' lies within a relative window w of an E4M3 rounding
midpoint.  w = 2^-14 covers the kernel's fp32 error in P' (about 2^-23 |S c|
from the FFMA, 2^-22 from ex2.approx, and the fp32 sum that forms S from exact
FP8 products) with a wide margin.  So, per output element,
  |dO_ic| <= sum_{j ambiguous} step_j |v_jc| v_descale / (2^8 l_i)
             + half a bf16 ulp of the reference + 1e-4 max|O|,
where step_j is the E4M3 spacing at P'_j: the result may take either
rounding there, and must be exact (to fp32 accumulation) elsewhere.
|dLSE| <= 1e-4.  P'_j is formed here from the oracle's definition: the
running max of the 128-key blocks up to j's block.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import online_softmax_sm_gb300 as fa
from tests import _parity as P

pytestmark = pytest.mark.gpu
W = 2.0 ** -14


def _e4m3_step(x):
    x = np.maximum(np.abs(x), 1e-300)
    e = np.floor(np.log2(x))
    return np.where(x < 2.0 ** -6, 2.0 ** -9, np.exp2(e - 3))


def _ambiguity(q, k, v, s_qk, vd, causal, block=128, rows=None):
    """Per row (all, or the listed query rows) and column: sum over keys whose
    P' sits near a rounding midpoint of (E4M3 step) |v| v_descale / (2^8 l)."""
    nq, nk = q.shape[0], k.shape[0]
    r = np.arange(nq) if rows is None else np.asarray(rows)
    s = s_qk * (q[r] @ k.T)
    if causal:
        i = r[:, None] + (nk - nq)
        s = np.where(np.arange(nk)[None, :] <= i, s, -np.inf)
    m_run = np.full((len(r), nk), -np.inf)
    m = np.full(len(r), -np.inf)
    for j0 in range(0, nk, block):
        m = np.maximum(m, s[:, j0:j0 + block].max(axis=1))
        m_run[:, j0:j0 + block] = m[:, None]
    with np.errstate(invalid="ignore", over="ignore"):
        pp = np.where(np.isfinite(s), np.exp2((s - m_run) * math.log2(math.e) + 8), 0.0)
    step = _e4m3_step(pp)
    frac = pp / step
    near = np.abs(frac - np.floor(frac) - 0.5) * step <= W * pp  # within w of a midpoint
    near &= pp > 0
    # l in the oracle's units: sum of P' against the final max, / 2^8
    m_fin = m[:, None]
    with np.errstate(invalid="ignore"):
        l = np.where(np.isfinite(s), np.exp(s - m_fin), 0.0).sum(axis=1)
    # a P' against a running max m_r enters O with weight exp(m_r - m_fin) after rescaling
    with np.errstate(invalid="ignore"):  # rows with no visible key: -inf - (-inf), discarded
        w = np.where(near, step * np.exp(np.where(np.isfinite(m_run), m_run - m_fin, 0.0)), 0.0)
    amb = (w @ np.abs(v)) * vd / (256.0 * np.where(l > 0, l, 1.0))[:, None]
    return amb


def _fp8(rng, shape, sd):
    return torch.tensor(rng.standard_normal(shape) * sd, dtype=torch.float32).to(torch.float8_e4m3fn)


def _check(q8, k8, v8, o, lse, scale, qd, kd, vd, causal, what, heads=None, rows=None):
    """Every head and row, or the listed (b, h) heads and query rows."""
    B, H = q8.shape[:2]
    heads = heads or [(b, h) for b in range(B) for h in range(H)]
    for b, h in heads:
        q, k, v = (t[b, h].float().cpu().double().numpy() for t in (q8, k8, v8))
        o_ref, l_ref = oracle.attention_fp8(q, k, v, scale, qd, kd, vd, causal=causal, rows=rows)
        og = o[b, h].cpu().double().numpy()
        lg = lse[b, h].cpu().double().numpy()
        if rows is not None:
            og, lg = og[rows], lg[rows]
        empty = np.isneginf(l_ref)
        assert np.all(og[empty] == 0) and np.all(np.isneginf(lg[empty])), what
        amb = _ambiguity(q, k, v, scale * qd * kd, vd, causal, rows=rows)
        tol = amb + P.half_ulp_bf16(o_ref) + 1e-4 * np.abs(o_ref).max(initial=0.0)
        err = np.abs(og - o_ref)
        bad = err > tol
        assert not bad.any(), (f"{what} (b={b},h={h}): {bad.sum()} of {bad.size} out of bound, worst "
                               f"excess {(err - tol).max():.3e}, max|dO| {err.max():.3e}")
        d = np.abs(lg[~empty] - l_ref[~empty])
        assert d.max(initial=0.0) <= 1e-4, f"{what}: max|dLSE| {d.max():.3e}"


# B, H, Nq, Nk, causal, sd (value spread)
CASES = [(1, 2, 256, 256, False, 1.0), (1, 2, 256, 256, True, 1.0), (1, 1, 200, 333, False, 2.0),
         (1, 2, 384, 129, True, 1.0), (2, 1, 130, 1000, False, 1.5), (1, 1, 512, 512, True, 3.0)]


@pytest.mark.parametrize("B,H,Nq,Nk,causal,sd", CASES,
                         ids=[f"b{c[0]}h{c[1]}nq{c[2]}nk{c[3]}{'c' if c[4] else 'n'}sd{c[5]}" for c in CASES])
def test_fp8_all_elements(B, H, Nq, Nk, causal, sd):
    rng = np.random.default_rng(Nq + Nk)
    q8, k8, v8 = (_fp8(rng, (B, H, n, 128), sd).cuda() for n in (Nq, Nk, Nk))
    scale, qd, kd, vd = 128 ** -0.5, 0.5, 0.75, 1.25
    o, lse = fa.fwd_fp8(q8, k8, v8, scale, qd, kd, vd, causal)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    _check(q8, k8, v8, o, lse, scale, qd, kd, vd, causal, f"{Nq}x{Nk} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_exact_when_every_p_is_representable(causal):
    """Q rows with eight ones, K rows with sixteen: every logit is an integer in
    [0, 8], so with scale = ln 2 every P' = 2^(s - m + 8) is a power of two in
    [1, 256] -- no E4M3 rounding decision -- and every alpha a power of two:
    the result is the exact attention of these inputs (fp64 oracle)."""
    rng = np.random.default_rng(9)
    B, H, N = 1, 2, 384

    def ones(rows, k):
        m = np.zeros((B, H, rows, 128), dtype=np.float32)
        for idx in np.ndindex(B, H, rows):
            m[idx][rng.choice(128, size=k, replace=False)] = 1.0
        return m

    q8 = torch.tensor(ones(N, 8)).to(torch.float8_e4m3fn).cuda()
    k8 = torch.tensor(ones(N, 16)).to(torch.float8_e4m3fn).cuda()
    v8 = torch.tensor(rng.integers(-4, 5, size=(B, H, N, 128)), dtype=torch.float32).to(
        torch.float8_e4m3fn).cuda()
    scale = math.log(2.0)
    o, lse = fa.fwd_fp8(q8, k8, v8, scale, 1.0, 1.0, 1.0, causal)
    torch.cuda.synchronize()
    for h in range(H):
        q, k, v = (t[0, h].float().double().cpu().numpy() for t in (q8, k8, v8))
        o_ref, l_ref = oracle.attention(q, k, v, scale, causal)
        og = o[0, h].cpu().double().numpy()
        tol = P.half_ulp_bf16(o_ref) + 1e-5 * np.abs(o_ref).max()
        assert np.all(np.abs(og - o_ref) <= tol), np.abs(og - o_ref).max()
        assert np.abs(lse[0, h].cpu().double().numpy() - l_ref).max() <= 1e-5


def test_fp8_rejects_other_head_dims():
    q8 = torch.zeros((1, 1, 128, 64), dtype=torch.float8_e4m3fn, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.fwd_fp8(q8, q8, q8, 0.125)
    assert e.value.code == fa.FA_ERR_UNSUPPORTED


@pytest.mark.parametrize("name", ["c3", "c4"])
def test_fp8_workload_sampled(name):
    """The benchmark's FP8 launches: the bf16 workload cast to E4M3, descales
    1, at full size; every tile's first and last row plus seeded extras of the
    first and last head."""
    from online_softmax_sm_gb300 import workloads

    w = workloads.C3 if name == "c3" else workloads.C4
    q8, k8, v8 = (t.to(torch.float8_e4m3fn) for t in workloads.generate(w, device="cuda"))
    o, lse = fa.fwd_fp8(q8, k8, v8, w.scale, 1.0, 1.0, 1.0, w.causal)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    rows = P.sample_rows(w.Nq, extra=64, seed=5)
    _check(q8, k8, v8, o, lse, w.scale, 1.0, 1.0, 1.0, w.causal, f"{w.name} fp8",
           heads=[(0, 0), (w.B - 1, w.H - 1)], rows=rows)
