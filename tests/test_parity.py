"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded bf16 inputs, element by element.  Tolerances in tests/_parity.py."""
import math

import numpy as np
import pytest
import torch

import oracle
import online_softmax_sm_gb300 as fa
from online_softmax_sm_gb300 import workloads
from tests import _parity as P

pytestmark = pytest.mark.gpu


# ------------------------------------------------------- small / ragged shapes

SMALL = [
    # B, H, Nq, Nk, d, causal, n_splits, bc, qt
    (1, 1, 1, 1, 64, False, 1, 0, 0),
    (1, 1, 1, 1, 128, False, 1, 0, 0),
    (1, 2, 63, 65, 64, False, 1, 0, 0),
    (1, 1, 129, 127, 128, False, 1, 0, 0),
    (2, 3, 200, 300, 128, False, 1, 0, 0),
    (1, 2, 256, 256, 64, False, 1, 64, 0),
    (1, 1, 384, 1000, 64, False, 1, 0, 0),
    (1, 2, 300, 300, 128, True, 1, 0, 0),
    (1, 1, 257, 129, 64, True, 1, 0, 0),      # Nq > Nk: fully masked rows
    (1, 1, 100, 1000, 128, True, 1, 0, 0),    # Nq < Nk
    (1, 1, 513, 513, 128, True, 1, 64, 0),
    (1, 2, 128, 1000, 128, False, 3, 0, 0),
    (2, 1, 300, 700, 64, False, 4, 0, 0),
    (1, 1, 200, 600, 128, True, 3, 0, 0),
    (1, 1, 330, 130, 128, True, 2, 0, 0),     # masked rows + splits (some splits empty)
    (1, 2, 256, 512, 128, False, 1, 0, 1),    # one Q tile per CTA forced
    (1, 2, 256, 512, 64, True, 1, 0, 1),
    (1, 1, 130, 260, 128, False, 1, 128, 2),  # two Q tiles per CTA, second ragged
    (1, 1, 64, 5000, 128, False, 1, 0, 0),
    (1, 1, 64, 5000, 128, False, 7, 64, 0),
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,n_splits,bc,qt", SMALL,
                         ids=[f"b{c[0]}h{c[1]}q{c[2]}k{c[3]}d{c[4]}{'c' if c[5] else ''}s{c[6]}bc{c[7]}qt{c[8]}"
                              for c in SMALL])
def test_small_shapes_all_rows(B, H, Nq, Nk, d, causal, n_splits, bc, qt):
    w = workloads.custom(B, H, Nq, Nk, d, seed=Nq * 7 + Nk, causal=causal, n_splits=n_splits, bc=bc,
                         q_mult=2.0)
    diff = P.run_workload(w, qt=qt)
    print(diff.check(w.name))


# Persistent grid: with at most 1-3 CTAs, each walks many work items, carrying
# TMEM, barrier phases, the K/V ring and the Q / staging buffers across them.
# Same arithmetic per item, so the result must equal the one-CTA-per-SM
# launch bit for bit, and match the oracle.
PERSIST = [
    # B, H, Nq, Nk, d, causal, n_splits, bc, qt
    (1, 3, 300, 700, 128, True, 1, 0, 0),
    (2, 3, 200, 300, 64, False, 1, 0, 0),
    (1, 2, 513, 513, 128, True, 1, 64, 0),
    (2, 1, 300, 700, 64, False, 4, 0, 0),
    (1, 1, 330, 130, 128, True, 2, 0, 0),     # masked rows, empty splits
    (1, 2, 256, 512, 64, True, 1, 0, 1),
    (1, 2, 257, 129, 64, True, 1, 0, 0),      # items whose tiles see no key
    (1, 2, 640, 900, 128, False, 1, 0, 0),
]


@pytest.mark.parametrize("max_ctas", [1, 2, 3])
@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,n_splits,bc,qt", PERSIST,
                         ids=[f"b{c[0]}h{c[1]}q{c[2]}k{c[3]}d{c[4]}{'c' if c[5] else ''}s{c[6]}bc{c[7]}qt{c[8]}"
                              for c in PERSIST])
def test_persistent_items_per_cta(B, H, Nq, Nk, d, causal, n_splits, bc, qt, max_ctas):
    w = workloads.custom(B, H, Nq, Nk, d, seed=Nq * 5 + Nk + max_ctas, causal=causal,
                         n_splits=n_splits, bc=bc, q_mult=2.0)
    q, k, v = workloads.generate(w, device="cuda")
    o0, l0 = fa.fwd(q, k, v, w.scale, causal, n_splits, bc=bc, q_tiles_per_cta=qt)
    o1 = torch.full_like(q, float("nan"))
    l1 = torch.full((B, H, Nq), float("nan"), device="cuda")
    fa.fwd(q, k, v, w.scale, causal, n_splits, out=o1, lse=l1, bc=bc, q_tiles_per_cta=qt,
           max_ctas=max_ctas)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    print(P.compare(q, k, v, o1, l1, w.scale, causal).check(f"{w.name} max_ctas={max_ctas}"))


def test_large_logits_and_growing_max():
    # Logits far above the fp16 overflow point and a running max that grows
    # along the key axis: exercises every rescale path.
    w = workloads.custom(1, 2, 256, 2048, 128, seed=5, q_mult=8.0, k_ramp=True)
    print(P.run_workload(w).check(w.name))


@pytest.mark.parametrize("bc", [64, 128])
def test_reference_moves_and_stays(bc):
    """Row maxima that grow by a set amount per K/V tile: with key j of tile t
    carrying g*t in dimension 0 and query row r carrying a_r there, row r's
    max grows by about a_r*g*log2(e) base-2 units per tile.  a_r spans 0.25..2
    with g*log2(e) = 12, so some rows grow by less than 16 units per tile (the
    kernel keeps its softmax reference for several tiles, P up to 2^16) and
    others by more (it moves the reference and rescales O on every tile)."""
    B, H, Nq, Nk, d = 1, 2, 256, 8 * 128, 64
    g = torch.Generator().manual_seed(11)
    q = 0.05 * torch.randn((B, H, Nq, d), generator=g)
    k = 0.05 * torch.randn((B, H, Nk, d), generator=g)
    v = torch.randn((B, H, Nk, d), generator=g)
    q[..., 0] = torch.linspace(0.25, 2.0, Nq)
    k[..., 0] = (torch.arange(Nk) // 128).float() * (12.0 / math.log2(math.e))
    q, k, v = (t.to(torch.bfloat16).cuda() for t in (q, k, v))
    o, lse = fa.fwd(q, k, v, 1.0, False, bc=bc)
    torch.cuda.synchronize()
    print(P.compare(q, k, v, o, lse, 1.0, False).check(f"reference moves/stays bc={bc}"))


# --------------------------------------------------- the pages' worked examples

def _example_case(scores_blocks, values, bc=64, n_splits=1):
    """Put each block of scores in its own K/V tile (scale 1, q = e0, k_j = s_j e0);
    pad the rest of each tile with keys of logit -200, whose exp is 0 in fp32."""
    d = 64
    nb = len(scores_blocks)
    Nk = bc * nb
    q = torch.zeros((1, 1, 1, d))
    q[0, 0, 0, 0] = 1.0
    k = torch.zeros((1, 1, Nk, d))
    k[0, 0, :, 0] = -200.0
    v = torch.zeros((1, 1, Nk, d))
    col = 0
    for b, blk in enumerate(scores_blocks):
        for t, s in enumerate(blk):
            k[0, 0, b * bc + t, 0] = s
            v[0, 0, b * bc + t] = torch.as_tensor(values[col], dtype=torch.float32)
            col += 1
    q, k, v = (x.to(torch.bfloat16).cuda() for x in (q, k, v))
    o, lse = fa.fwd(q, k, v, 1.0, False, n_splits, bc=bc)
    torch.cuda.synchronize()
    return q, k, v, o, lse


@pytest.mark.parametrize("n_splits", [1, 2])
@pytest.mark.parametrize("bc", [64, 128])
def test_worked_examples_through_gpu(n_splits, bc):
    d = 64
    onehot = [np.eye(d)[i] for i in range(4)]
    # [2,4] then [1,3]: l = 1.553, m = 4 (no rescale)
    q, k, v, o, lse = _example_case([[2, 4], [1, 3]], onehot, bc, n_splits)
    l = math.exp(float(lse[0, 0, 0]) - 4.0)
    assert abs(l - 1.553) <= 1e-3
    p_exact = np.exp(np.array([2, 4, 1, 3]) - 4.0) / l
    np.testing.assert_allclose(o[0, 0, 0, :4].float().cpu().numpy(), p_exact, rtol=0, atol=4e-3)
    # [1,2] then [5,3]: m = 5, l = 1.2034 (rescale in the second tile)
    q, k, v, o, lse = _example_case([[1, 2], [5, 3]], onehot, bc, n_splits)
    assert abs(math.exp(float(lse[0, 0, 0]) - 5.0) - 1.2034) <= 1e-4
    P.compare(q, k, v, o, lse, 1.0, False).check("p1 rescale example")
    # s = [1,2,3,10], V = 1: O = 1, l = 1.00137
    ones = [np.ones(d)] * 4
    q, k, v, o, lse = _example_case([[1, 2], [3, 10]], ones, bc, n_splits)
    assert abs(math.exp(float(lse[0, 0, 0]) - 10.0) - 1.00137) <= 1e-5
    assert torch.all(o[0, 0, 0] == 1.0)


def test_scores_order_and_block_independence():
    # Reversing the key order (and the values with it) must not change O or LSE
    # beyond rounding: the recurrence is order independent.
    w = workloads.custom(1, 2, 128, 1500, 128, seed=9, q_mult=3.0)
    q, k, v = workloads.generate(w, device="cuda")
    o1, l1 = fa.fwd(q, k, v, w.scale)
    o2, l2 = fa.fwd(q, k.flip(2).contiguous(), v.flip(2).contiguous(), w.scale)
    torch.cuda.synchronize()
    assert (o1.float() - o2.float()).abs().max().item() <= 8e-3
    assert (l1 - l2).abs().max().item() <= 2e-4


# ----------------------------------------------------------- robustness checks

def test_deterministic_and_fully_overwrites():
    w = workloads.custom(2, 4, 500, 700, 128, seed=11, causal=True)
    q, k, v = workloads.generate(w, device="cuda")
    o1 = torch.full_like(q, float("nan"))
    l1 = torch.full((2, 4, 500), float("nan"), device="cuda")
    fa.fwd(q, k, v, w.scale, True, out=o1, lse=l1)
    o2, l2 = fa.fwd(q, k, v, w.scale, True)
    torch.cuda.synchronize()
    assert not torch.isnan(o1).any() and not torch.isnan(l1).any()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_shift_invariance_on_gpu():
    # softmax(s + c) = softmax(s): a last feature a (queries) times b (keys)
    # adds scale*a*b to every logit, so O is unchanged and LSE moves by it.
    w = workloads.custom(1, 1, 256, 384, 64, seed=12)
    q, k, v = workloads.generate(w, device="cuda")
    q0, k0 = q.clone(), k.clone()
    q0[..., -1] = 0.0
    k0[..., -1] = 0.0
    q2, k2 = q0.clone(), k0.clone()
    q2[..., -1] = 4.0  # exact in bf16
    k2[..., -1] = 2.0
    o0, l0 = fa.fwd(q0, k0, v, 0.5)
    o2, l2 = fa.fwd(q2, k2, v, 0.5)
    torch.cuda.synchronize()
    assert (o0.float() - o2.float()).abs().max().item() <= 8e-3
    assert ((l2 - l0) - 4.0).abs().max().item() <= 1e-3


# --------------------------------------------------------- the five workloads

def test_c1_all_rows_bc64():
    print(P.run_workload(workloads.C1).check("C1"))


def test_c2_all_rows():
    print(P.run_workload(workloads.C2).check("C2"))


def test_c3_every_row():
    """All B*H*Nq = 262144 rows of C3 against the oracle (about 10 s of host time)."""
    w = workloads.C3
    d = P.run_workload(w)
    assert d.rows == w.B * w.H * w.Nq
    print(d.check("C3"))


def test_c4_causal_every_row():
    """All B*H*Nq = 524288 rows of C4 (causal, 16K) against the oracle (about half a minute of
    host time on 16 cores)."""
    w = workloads.C4
    d = P.run_workload(w)
    assert d.rows == w.B * w.H * w.Nq
    print(d.check("C4"))


def test_c4_companion_fully_masked_rows():
    w = workloads.C4_MASKED
    q, k, v = workloads.generate(w, device="cuda")
    o, lse = fa.fwd(q, k, v, w.scale, True)
    torch.cuda.synchronize()
    # rows 0..255 see no key under bottom-right alignment (Nk = Nq - 256)
    assert torch.all(o[:, :, :256] == 0)
    assert torch.all(torch.isneginf(lse[:, :, :256]))
    assert torch.isfinite(lse[:, :, 256:]).all()
    rows = list(range(0, 260)) + P.sample_rows(w.Nq, extra=64, seed=4)
    P.compare(q, k, v, o, lse, w.scale, True, heads=[(0, 2), (0, 30)], rows=sorted(set(rows))).check("C4 masked")


def test_c5_split_kv_every_row():
    """All B*H*Nq = 65536 rows of C5 (16 splits, merged) against the oracle."""
    w = workloads.C5
    d = P.run_workload(w)
    assert d.rows == w.B * w.H * w.Nq
    print(d.check("C5"))


def test_c5_split_equals_unsplit():
    w = workloads.custom(2, 4, 128, 32768, 128, seed=21)
    q, k, v = workloads.generate(w, device="cuda")
    o1, l1 = fa.fwd(q, k, v, w.scale, False, 16)
    o2, l2 = fa.fwd(q, k, v, w.scale, False, 1)
    torch.cuda.synchronize()
    assert (o1.float() - o2.float()).abs().max().item() <= 8e-3
    assert (l1 - l2).abs().max().item() <= 5e-4
