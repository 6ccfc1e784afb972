"""GPU parity of the split-KV pieces: fa_fwd_partial against the oracle on each
split's key range, and fa_merge_splits against the oracle's two-block merge
rule (folded pairwise) on random partial triples, empty splits included."""
import math

import numpy as np
import pytest
import torch

import oracle
import online_softmax_sm_gb300 as fa
from online_softmax_sm_gb300 import workloads
from tests import _parity as P

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("S", [1, 2, 5, 16])
def test_merge_kernel_matches_oracle_merge(d, S):
    rng = np.random.default_rng(100 * S + d)
    B, H, Nq = 2, 3, 37
    m = rng.standard_normal((S, B, H, Nq)) * 6
    l = rng.uniform(0.5, 40.0, size=(S, B, H, Nq))
    # partial O rows are softmax-weighted means of V rows, so of magnitude well
    # below 1; N(0,1)*0.3 keeps bf16 output rounding (relative 2^-9) under the bar
    o = rng.standard_normal((S, B, H, Nq, d)) * 0.3
    # empty splits: m = -inf, l = 0, O = 0 (a whole row empty when S == 1 for row 0)
    empty = rng.random((S, B, H, Nq)) < 0.25
    empty[:, 0, 0, 0] = True
    m[empty] = -np.inf
    l[empty] = 0.0
    o[empty] = 0.0
    mt, lt, ot = (torch.as_tensor(x, dtype=torch.float32).cuda().contiguous() for x in (m, l, o))
    out, lse = fa.merge_splits(mt, lt, ot)
    torch.cuda.synchronize()
    m32, l32, o32 = (x.cpu().double().numpy() for x in (mt, lt, ot))  # what the GPU saw
    diff = P.Diff()
    for b in range(B):
        for h in range(H):
            o_ref = np.empty((Nq, d))
            lse_ref = np.empty(Nq)
            for i in range(Nq):
                _, _, o_ref[i], lse_ref[i] = oracle.merge(m32[:, b, h, i], l32[:, b, h, i], o32[:, b, h, i])
            diff.add(out[b, h].cpu().double().numpy(), lse[b, h].cpu().double().numpy(), o_ref, lse_ref)
    assert diff.masked_rows >= 1
    print(diff.check(f"merge S={S} d={d}"))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d,Nq,Nk,S", [(128, 128, 1000, 3), (64, 200, 777, 4), (128, 300, 300, 5)])
def test_partial_triples_match_oracle_per_split(causal, d, Nq, Nk, S):
    w = workloads.custom(1, 2, Nq, Nk, d, seed=Nk + S, causal=causal, q_mult=2.0)
    q, k, v = workloads.generate(w, device="cuda")
    m_p, l_p, o_p = fa.fwd_partial(q, k, v, S, w.scale, causal)
    torch.cuda.synchronize()
    T = math.ceil(Nk / 128)
    per = math.ceil(T / S)
    for s in range(S):
        k0, k1 = min(s * per * 128, Nk), min((s + 1) * per * 128, Nk)
        for h in range(2):
            mm = m_p[s, 0, h].cpu().double().numpy()
            ll = l_p[s, 0, h].cpu().double().numpy()
            oo = o_p[s, 0, h].cpu().double().numpy()
            lse_gpu = np.where(ll > 0, mm + np.log(np.where(ll > 0, ll, 1.0)), -np.inf)
            if k1 <= k0:  # split past the end of the key axis: empty
                assert np.all(np.isneginf(mm)) and np.all(ll == 0) and np.all(oo == 0)
                continue
            # keys [k0, k1) of this split; causal visibility keeps the global offset
            qh, kh, vh = q[0, h].cpu(), k[0, h, k0:k1].cpu(), v[0, h, k0:k1].cpu()
            o_ref = np.zeros((Nq, d))
            lse_ref = np.full(Nq, -np.inf)
            if causal:
                # visible iff j <= i + (Nk - Nq), j global; in the slice j = k0 + jj
                kq = kh.double().numpy()
                vq = vh.double().numpy()
                qq = qh.double().numpy()
                for i in range(Nq):
                    last = i + (Nk - Nq) - k0
                    if last < 0:
                        continue
                    cnt = min(last + 1, k1 - k0)
                    oi, li = oracle.attention(qq[i:i + 1], kq[:cnt], vq[:cnt], w.scale, False)
                    o_ref[i], lse_ref[i] = oi[0], li[0]
            else:
                o_ref, lse_ref = oracle.attention(qh, kh, vh, w.scale, False)
            diff = P.Diff()
            diff.add(oo, lse_gpu, o_ref, lse_ref)
            diff.check(f"split {s} head {h}")


def test_partial_plus_merge_equals_fwd():
    """fa_fwd's split path is fa_fwd_partial + fa_merge_splits with O_s kept
    in bf16 in its own workspace: merging the public fp32 partials after
    rounding O_s to bf16 (round to nearest even, as the kernel does; the merge
    upcasts exactly) gives fa_fwd's O and LSE bit for bit, and the fp32
    partials themselves differ from it by at most the bf16 rounding of O_s."""
    w = workloads.custom(2, 2, 256, 3000, 128, seed=77, causal=True)
    q, k, v = workloads.generate(w, device="cuda")
    m_p, l_p, o_p = fa.fwd_partial(q, k, v, 6, w.scale, True)
    o_bf = o_p.to(torch.bfloat16).to(torch.float32).contiguous()
    o1, l1 = fa.merge_splits(m_p, l_p, o_bf)
    o32, l32 = fa.merge_splits(m_p, l_p, o_p)
    o2, l2 = fa.fwd(q, k, v, w.scale, True, 6)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)
    ninf = lambda t: torch.nan_to_num(t, neginf=-1e30)
    assert torch.equal(ninf(l1), ninf(l2)) and torch.equal(ninf(l32), ninf(l2))
    # |O(bf16 partials) - O(fp32 partials)| <= 2^-8 max_s |O_s| + one bf16 step of O
    bound = 2.0 ** -8 * o_p.abs().amax(dim=0) + 2.0 ** -7 * o32.float().abs() + 1e-30
    assert ((o2.float() - o32.float()).abs() <= bound).all()
