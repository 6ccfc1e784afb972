"""Pins for the fp64 oracle, independent of the oracle itself.

Each test checks the oracle against something the pages or mathematics fix:
values printed for worked examples (tests/golden/worked_examples.json, each
with its citation), closed forms, invariants the pages state, special cases
that reduce to library routines (scipy.special.softmax / logsumexp), and the
masked-row convention.  tests/test_oracle_mutants.py checks that plausible
mistakes in oracle.c fail at least one of these pins.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special as sps

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")


@pytest.fixture(scope="module")
def golden():
    with open(GOLDEN, encoding="utf-8") as f:
        return json.load(f)


def close(a, b, unit):
    return abs(float(a) - float(b)) <= unit * (1 + 1e-9)


def one_row_attention(scores, values, scale=1.0, causal=False):
    """Feed a score row through the attention routine: q = e0, k_j = s_j e0."""
    s = np.asarray(scores, dtype=np.float64)
    v = np.asarray(values, dtype=np.float64)
    if v.ndim == 1:
        v = v[:, None]
    n, dv = v.shape
    d = max(dv, 1)
    q = np.zeros((1, d))
    q[0, 0] = 1.0
    k = np.zeros((n, d))
    k[:, 0] = s
    vv = np.zeros((n, d))
    vv[:, :dv] = v
    o, lse = oracle.attention(q, k, vv, scale, causal)
    return o[0, :dv], lse[0]


# ---------------------------------------------------------------- worked examples

def test_p1_no_rescale_example(golden):
    g = golden["p1_no_rescale"]
    s, blocks = g["scores"], [tuple(b) for b in g["blocks"]]
    m1, l1, _, _ = oracle.online_blocks(s[:2], np.ones(2), [(0, 2)])
    assert m1 == g["after_block_1"]["m"] and close(l1, g["after_block_1"]["l"], g["after_block_1"]["unit"])
    for x, p in zip(s[2:], g["block_2_exps"]["values"]):
        assert close(math.exp(x - m1), p, g["block_2_exps"]["unit"])
    m, l, o, lse = oracle.online_blocks(s, np.ones(4), blocks)
    assert m == g["final"]["m"] and close(l, g["final"]["l"], g["final"]["unit"])
    assert abs(o[0] - 1.0) < 1e-15
    # the same through the three-pass attention routine
    o_att, lse_att = one_row_attention(s, np.ones(4))
    assert abs(lse_att - lse) < 1e-13 and abs(lse - (m + math.log(l))) < 1e-15


def test_p1_rescale_example(golden):
    g = golden["p1_rescale"]
    s, blocks = g["scores"], [tuple(b) for b in g["blocks"]]
    m1, l1, _, _ = oracle.online_blocks(s[:2], np.ones(2), [(0, 2)])
    assert m1 == g["after_block_1"]["m"] and close(l1, g["after_block_1"]["l"], g["after_block_1"]["unit"])
    alpha = math.exp(m1 - 5.0)
    assert close(alpha, g["second_block_scale"]["value"], g["second_block_scale"]["unit"])
    assert close(l1 * alpha, g["scaled_l"]["value"], g["scaled_l"]["unit"])
    m, l, _, _ = oracle.online_blocks(s, np.ones(4), blocks)
    assert m == g["final"]["m"]
    assert close(l, g["final"]["l"], g["final"]["unit"])
    assert close(l, g["check_sum"]["total"], g["check_sum"]["unit"])
    # the page's per-term check: exp(s_j - 5) for each score
    for x, t in zip(s, [g["check_sum"]["terms"][i] for i in (0, 1, 2, 3)]):
        assert close(math.exp(x - 5.0), t, g["check_sum"]["unit"])
    # block order reversed gives the same state
    m_r, l_r, _, _ = oracle.online_blocks(s, np.ones(4), blocks[::-1])
    assert m_r == m and abs(l_r - l) < 1e-14


def test_p4_large_jump_example(golden):
    g = golden["p4_large_jump"]
    s, v, blocks = g["scores"], g["values"], [tuple(b) for b in g["blocks"]]
    m1, l1, o1, _ = oracle.online_blocks(s[:2], v[:2], [(0, 2)])
    a1 = g["after_block_1"]
    assert m1 == a1["m"] and close(l1, a1["l"], a1["unit"])
    assert close(o1[0] * l1, a1["o_unnormalised"], a1["unit"])  # unnormalised O
    for x, p in zip(s[:2], a1["p"]):
        assert close(math.exp(x - m1), p, a1["unit"])
    alpha = math.exp(m1 - 10.0)
    assert close(alpha, g["alpha"]["value"], g["alpha"]["unit"])
    assert close(alpha * l1, g["rescaled_l"]["value"], g["rescaled_l"]["unit"])
    for x, p in zip(s[2:], g["p_2"]["values"]):
        assert close(math.exp(x - 10.0), p, g["p_2"]["unit"])
    m, l, o, _ = oracle.online_blocks(s, v, blocks)
    assert m == g["final"]["m"] and close(l, g["final"]["l"], g["final"]["unit"])
    assert abs(o[0] - g["final"]["o"]) < 1e-15
    sa = g["softmax_all_at_once"]
    p_att, _ = one_row_attention(s, np.eye(4))
    for pv, ref, unit, garbled in zip(p_att, sa["values"], sa["units"], sa["garbled"]):
        if garbled:
            assert abs(pv - ref) <= sa["garbled_rel_tol"] * ref
        else:
            assert close(pv, ref, unit)


def test_p1_overflow_row(golden):
    g = golden["p1_overflow_row"]
    s = np.array(g["scores"], dtype=np.float64)
    p, lse = one_row_attention(s, np.eye(3))
    assert np.all(np.isfinite(p)) and abs(p.sum() - 1.0) < 1e-15
    # LSE from the page's printed exponentials, within their printed precision
    lse_printed = math.log(sum(g["printed_exp"]))
    assert abs(lse - lse_printed) <= g["printed_exp_rel_unit"]
    # each P_j against the printed exp_j / sum(printed)
    for pj, e in zip(p, g["printed_exp"]):
        assert abs(pj - e / sum(g["printed_exp"])) <= 2 * g["printed_exp_rel_unit"] * pj
    # fp64 exp overflows above ~709.78; the stable form must not
    p2, lse2 = one_row_attention([1000.0, 1001.0], np.eye(2))
    assert abs(p2[0] - 1 / (1 + math.e)) < 1e-15 and abs(p2[1] - math.e / (1 + math.e)) < 1e-15
    assert abs(lse2 - (1001.0 + math.log1p(math.exp(-1.0)))) < 1e-12


def test_p4_practice_1_closed_form():
    # s = [0] then [5], V = [[2],[3]].  Closed form: O = (2 e^-5 + 3) / (1 + e^-5),
    # l = 1 + e^-5 relative to m = 5.
    m, l, o, lse = oracle.online_blocks([0.0, 5.0], [[2.0], [3.0]], [(0, 1), (1, 1)])
    e5 = math.exp(-5.0)
    assert m == 5.0 and abs(l - (1 + e5)) < 1e-15
    assert abs(o[0] - (2 * e5 + 3) / (1 + e5)) < 1e-15
    assert abs(lse - (5 + math.log1p(e5))) < 1e-15


def test_first_block_from_minus_inf():
    # Starting state m = -inf, l = 0: the first block's scale exp(-inf - m') is 0
    # and no NaN appears, also when a whole block is -inf.
    ninf = -math.inf
    s = [ninf, ninf, 1.0, 2.0]
    m, l, o, lse = oracle.online_blocks(s, np.eye(4), [(0, 2), (2, 2)])
    assert m == 2.0 and abs(l - (1 + math.exp(-1))) < 1e-15
    assert np.all(np.isfinite(o)) and o[0] == 0.0 and o[1] == 0.0
    m, l, o, lse = oracle.online_blocks([ninf, ninf], np.eye(2), [(0, 1), (1, 1)])
    assert m == ninf and l == 0.0 and np.all(o == 0.0) and lse == ninf


# ------------------------------------------------------- library special cases

@pytest.mark.parametrize("nq,nk,d,causal,seed", [
    (5, 7, 3, False, 0), (7, 7, 4, True, 1), (4, 9, 2, True, 2),
    (9, 4, 3, True, 3), (1, 1, 5, False, 4), (3, 16, 8, False, 5),
])
def test_attention_matches_scipy_softmax(nq, nk, d, causal, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((nq, d)) * 2
    k = rng.standard_normal((nk, d))
    v = rng.standard_normal((nk, d))
    scale = 1 / math.sqrt(d)
    o, lse = oracle.attention(q, k, v, scale, causal)
    S = scale * (q @ k.T)
    if causal:
        ii = np.arange(nq)[:, None]
        jj = np.arange(nk)[None, :]
        S = np.where(jj <= ii + (nk - nq), S, -np.inf)
    for i in range(nq):
        if np.all(np.isneginf(S[i])):
            assert np.all(o[i] == 0.0) and lse[i] == -np.inf
            continue
        p = sps.softmax(S[i])
        np.testing.assert_allclose(o[i], p @ v, rtol=1e-12, atol=1e-13)
        assert abs(lse[i] - sps.logsumexp(S[i])) < 1e-12


def test_rows_subset_and_threads_agree():
    rng = np.random.default_rng(7)
    q, k, v = (rng.standard_normal((33, 16)) for _ in range(3))
    o_all, l_all = oracle.attention(q, k, v, 0.25, True, threads=1)
    rows = [32, 0, 5, 5, 17]
    o_sub, l_sub = oracle.attention(q, k, v, 0.25, True, rows=rows, threads=3)
    np.testing.assert_array_equal(o_sub, o_all[rows])
    np.testing.assert_array_equal(l_sub, l_all[rows])


def test_two_pass_softmax_matches_scipy():
    rng = np.random.default_rng(3)
    for n in (1, 2, 17, 300):
        x = rng.standard_normal(n) * 30
        p, lse = oracle.softmax_two_pass(x)
        np.testing.assert_allclose(p, sps.softmax(x), rtol=1e-12, atol=1e-300)
        assert abs(lse - sps.logsumexp(x)) < 1e-12
    p, lse = oracle.softmax_two_pass([-math.inf] * 3)
    assert np.all(p == 0) and lse == -math.inf


def test_softmax_rows_matches_scipy_rowwise():
    """The two-pass normaliser over a matrix ("Online Softmax 算法详解"
    section 2.2, row by row): scipy's softmax / logsumexp along axis 1, with
    -inf entries, an all -inf row (p = 0, lse = -inf) and a row shifted by
    1e4 (no overflow: exp is taken against the running max)."""
    rng = np.random.default_rng(11)
    for rows, cols in ((1, 1), (7, 33), (16, 257)):
        x = rng.standard_normal((rows, cols)) * 20
        x[rows // 2, :: 3] = -math.inf
        if rows > 2:
            x[1, :] = -math.inf
            x[2, :] += 1e4
        p, lse = oracle.softmax_rows(x, threads=3)
        live = ~np.all(np.isneginf(x), axis=1)
        np.testing.assert_allclose(p[live], sps.softmax(x[live], axis=1), rtol=1e-12, atol=1e-300)
        np.testing.assert_allclose(lse[live], sps.logsumexp(x[live], axis=1), rtol=1e-14, atol=1e-11)
        assert np.all(p[~live] == 0) and np.all(np.isneginf(lse[~live]))


def test_softmax_rows_selection():
    """A row selection returns exactly those rows, in the order given."""
    rng = np.random.default_rng(12)
    x = rng.standard_normal((9, 40)) * 5
    p_all, l_all = oracle.softmax_rows(x, threads=2)
    sel = [8, 0, 3, 3]
    p_sub, l_sub = oracle.softmax_rows(x, rows=sel, threads=4)
    np.testing.assert_array_equal(p_sub, p_all[sel])
    np.testing.assert_array_equal(l_sub, l_all[sel])
    np.testing.assert_allclose(p_sub, sps.softmax(x[sel], axis=1), rtol=1e-12)


# ------------------------------------------------------------- FP8 forward

def _torch_e4m3(x):
    """torch's float8_e4m3fn cast of x given as float32 values (torch casts
    through float32, so only float32 inputs are rounded exactly once)."""
    import torch
    x32 = np.asarray(x, dtype=np.float64).astype(np.float32)
    return torch.tensor(x32).to(torch.float8_e4m3fn).double().numpy()


def test_e4m3_rounding_matches_torch():
    """oracle_e4m3 against torch's float8_e4m3fn cast on [0, 448]: random
    values, every representable value, every midpoint (ties to even) and the
    subnormal range."""
    rng = np.random.default_rng(31)
    grid = np.unique(_torch_e4m3(np.linspace(0, 448, 20000)))
    mids = ((grid[1:] + grid[:-1]) / 2).astype(np.float32)
    x = np.concatenate([rng.uniform(0, 448, 5000), rng.uniform(0, 0.02, 2000), grid, mids,
                        np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1000))])
    x = x.astype(np.float32).astype(np.float64)  # float32-representable inputs
    np.testing.assert_array_equal(oracle.e4m3(x), _torch_e4m3(x))
    np.testing.assert_array_equal(oracle.e4m3(-x), -_torch_e4m3(x))


def _e4m3_values(rng, shape, scale):
    return _torch_e4m3(rng.standard_normal(shape) * scale)


def test_fp8_single_block_closed_form():
    """With one key block the running max is the row max: P' = 256 exp(s - m)
    exactly, O = sum_j E4M3(P'_j) v_j v_descale / sum_j P'_j, LSE = logsumexp(s)
    (torch's E4M3 cast and scipy's logsumexp)."""
    rng = np.random.default_rng(32)
    nq, nk, d = 6, 50, 8
    q, k, v = (_e4m3_values(rng, (n, d), 2.0) for n in (nq, nk, nk))
    scale, qd, kd, vd = 0.3, 0.5, 1.25, 0.75
    o, lse = oracle.attention_fp8(q, k, v, scale, qd, kd, vd, block=64)
    s_ = scale * qd * kd * (q @ k.T)
    pp = 256.0 * np.exp(s_ - s_.max(axis=1, keepdims=True))
    o_ref = (_torch_e4m3(pp) @ v) * vd / pp.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse, sps.logsumexp(s_, axis=1), rtol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_exact_when_every_p_is_representable(causal):
    """Integer logits with scale = ln 2 make every P' = 2^(s - m + 8) a power of
    two inside the E4M3 range and every alpha a power of two: the FP8 steps then
    lose nothing, and O, LSE equal the fp64 attention oracle (several blocks)."""
    rng = np.random.default_rng(33)
    nq, nk, d = 40, 70, 4
    q = rng.integers(-1, 2, size=(nq, d)).astype(np.float64)
    k = rng.integers(-1, 2, size=(nk, d)).astype(np.float64)
    v = _e4m3_values(rng, (nk, d), 1.0)
    o8, l8 = oracle.attention_fp8(q, k, v, math.log(2.0), causal=causal, block=16)
    o, lse = oracle.attention(q, k, v, math.log(2.0), causal)
    np.testing.assert_allclose(o8, o, rtol=1e-13, atol=1e-15)
    fin = np.isfinite(lse)
    np.testing.assert_array_equal(np.isfinite(l8), fin)
    np.testing.assert_allclose(l8[fin], lse[fin], rtol=1e-13)


def test_fp8_descales_are_scalings():
    """Doubling the E4M3 values of Q while halving q_descale (and the same for
    V) changes nothing."""
    rng = np.random.default_rng(34)
    q, k, v = (_e4m3_values(rng, (n, 8), 1.0) for n in (20, 300, 300))
    a = oracle.attention_fp8(q, k, v, 0.35, 1.0, 1.0, 1.0, block=128)
    b = oracle.attention_fp8(2 * q, k, 2 * v, 0.35, 0.5, 1.0, 0.5, block=128)
    np.testing.assert_allclose(a[0], b[0], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(a[1], b[1], rtol=1e-14)


# ------------------------------------------------------------- backward

def _loss_grads_fd(q, k, v, g, scale, window, h=1e-6):
    """Central differences of L = sum(O * g) through the forward oracle."""
    def loss(q_, k_, v_):
        o, _ = oracle.attention_window(q_, k_, v_, scale, window[0], window[1])
        return float(np.sum(o * g))
    out = []
    for which, arr in enumerate((q, k, v)):
        grad = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            hi, lo = [x.copy() for x in (q, k, v)], [x.copy() for x in (q, k, v)]
            hi[which][idx] += h
            lo[which][idx] -= h
            grad[idx] = (loss(*hi) - loss(*lo)) / (2 * h)
        out.append(grad)
    return out


@pytest.mark.parametrize("nq,nk,d,window,seed", [
    (3, 4, 2, (-1, -1), 0), (4, 4, 3, (-1, 0), 1), (5, 3, 2, (-1, 0), 2), (4, 6, 2, (1, 1), 3),
    (6, 5, 3, (2, 0), 4)])
def test_bwd_matches_finite_differences(nq, nk, d, window, seed):
    """Gradients of sum(O * dO) against central differences of the forward
    oracle (pinned independently above); includes masks that leave a row
    with no visible key."""
    rng = np.random.default_rng(seed)
    q, k, v, g = (rng.standard_normal(sh) for sh in ((nq, d), (nk, d), (nk, d), (nq, d)))
    scale = 0.8
    r = oracle.attention_bwd(q, k, v, g, scale, window=window)
    dq, dk, dv = _loss_grads_fd(q, k, v, g, scale, window)
    np.testing.assert_allclose(r["dq"], dq, rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(r["dk"], dk, rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(r["dv"], dv, rtol=1e-6, atol=1e-8)


def test_bwd_invariants_and_statistics():
    """sum_j dK_j = 0 and sum_j dV_j = sum of dO over rows that see a key
    (softmax rows sum to one); D_i = <dO_i, O_i>; LSE equals the forward's."""
    rng = np.random.default_rng(21)
    nq, nk, d = 9, 7, 4
    q, k, v, g = (rng.standard_normal(sh) for sh in ((nq, d), (nk, d), (nk, d), (nq, d)))
    for causal in (False, True):
        r = oracle.attention_bwd(q, k, v, g, 0.5, causal=causal, threads=3)
        o, lse = oracle.attention(q, k, v, 0.5, causal)
        live = np.isfinite(lse)
        np.testing.assert_allclose(r["dk"].sum(axis=0), 0.0, atol=1e-12)
        np.testing.assert_allclose(r["dv"].sum(axis=0), g[live].sum(axis=0), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(r["dd"][live], np.sum(g * o, axis=1)[live], rtol=1e-12, atol=1e-12)
        np.testing.assert_array_equal(np.isfinite(r["lse"]), live)
        np.testing.assert_allclose(r["lse"][live], lse[live], rtol=1e-14)
        assert np.all(r["dq"][~live] == 0.0)


def test_bwd_single_key():
    """One key: P = 1, so dS = 0 (dQ = dK = 0) and dV = sum_i dO_i."""
    rng = np.random.default_rng(22)
    q, g = rng.standard_normal((5, 3)), rng.standard_normal((5, 3))
    k, v = rng.standard_normal((1, 3)), rng.standard_normal((1, 3))
    r = oracle.attention_bwd(q, k, v, g, 1.3)
    assert np.abs(r["dq"]).max() < 1e-15 and np.abs(r["dk"]).max() < 1e-15
    np.testing.assert_allclose(r["dv"][0], g.sum(axis=0), rtol=1e-14)


# ------------------------------------------------------------- closed forms

def test_single_key():
    # Nk = 1: O = v_0 and LSE = scale * <q, k_0>.
    rng = np.random.default_rng(11)
    q, k, v = rng.standard_normal((4, 6)), rng.standard_normal((1, 6)), rng.standard_normal((1, 6))
    o, lse = oracle.attention(q, k, v, 0.5, False)
    np.testing.assert_array_equal(o, np.repeat(v, 4, axis=0))
    np.testing.assert_allclose(lse, 0.5 * (q @ k[0]), rtol=0, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_average_visible_values(causal):
    # Q = 0: P is uniform over the visible keys, O = their mean, LSE = ln(count).
    rng = np.random.default_rng(12)
    nq, nk, d = 6, 10, 4
    q = np.zeros((nq, d))
    k, v = rng.standard_normal((nk, d)), rng.standard_normal((nk, d))
    o, lse = oracle.attention(q, k, v, 0.3, causal)
    for i in range(nq):
        cnt = (i + nk - nq + 1) if causal else nk
        np.testing.assert_allclose(o[i], v[:cnt].mean(axis=0), rtol=1e-13, atol=1e-14)
        assert abs(lse[i] - math.log(cnt)) < 1e-14


def test_rows_of_p_sum_to_one_and_constant_values():
    # V = identity gives O = P (rows sum to 1); V = 1 gives O = 1.
    rng = np.random.default_rng(13)
    nk = 12
    q, k = rng.standard_normal((5, nk)) * 3, rng.standard_normal((nk, nk))
    o, _ = oracle.attention(q, k, np.eye(nk), 1.0, False)
    np.testing.assert_allclose(o.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    assert np.all(o > 0)
    o1, _ = oracle.attention(q, k, np.ones((nk, nk)), 1.0, True)
    np.testing.assert_allclose(o1, 1.0, rtol=0, atol=1e-14)


def test_shift_invariance():
    # Adding c to a row's logits (extra feature: q' = [q, c/scale], k' = [k, 1])
    # leaves O unchanged and shifts LSE by c.
    rng = np.random.default_rng(14)
    nq, nk, d, scale, c = 4, 9, 5, 0.7, 3.25
    q, k, v = rng.standard_normal((nq, d)), rng.standard_normal((nk, d)), rng.standard_normal((nk, d))
    o, lse = oracle.attention(q, k, v, scale, False)
    q2 = np.concatenate([q, np.full((nq, 1), c / scale)], axis=1)
    k2 = np.concatenate([k, np.ones((nk, 1))], axis=1)
    v2 = np.concatenate([v, np.zeros((nk, 1))], axis=1)
    o2, lse2 = oracle.attention(q2, k2, v2, scale, False)
    np.testing.assert_allclose(o2[:, :d], o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse2, lse + c, rtol=0, atol=1e-12)


def test_fully_masked_rows():
    # Causal with nq > nk: rows i < nq - nk see no key: O = 0 exactly, LSE = -inf.
    rng = np.random.default_rng(15)
    nq, nk, d = 8, 3, 4
    q, k, v = rng.standard_normal((nq, d)), rng.standard_normal((nk, d)), rng.standard_normal((nk, d))
    o, lse = oracle.attention(q, k, v, 1.0, True)
    for i in range(nq - nk):
        assert np.all(o[i] == 0.0) and lse[i] == -np.inf
    for i in range(nq - nk, nq):
        assert np.all(np.isfinite(o[i])) and np.isfinite(lse[i])
    # first visible row sees exactly key 0
    np.testing.assert_array_equal(o[nq - nk], v[0])


# ------------------------------------- block size / order independence, merge

@pytest.mark.parametrize("seed", [0, 1, 2])
def test_online_blocks_match_three_pass(seed):
    rng = np.random.default_rng(100 + seed)
    nk, d = 130, 5
    q = rng.standard_normal((1, d)) * 4
    k, v = rng.standard_normal((nk, d)), rng.standard_normal((nk, d))
    scale = 0.9
    o_ref, lse_ref = oracle.attention(q, k, v, scale, False)
    s = scale * (k @ q[0])
    for bc in (1, 2, 3, 64, 128, nk):
        blocks = [(j, min(bc, nk - j)) for j in range(0, nk, bc)]
        for order in range(3):
            bl = list(blocks)
            if order == 1:
                bl = bl[::-1]
            elif order == 2:
                rng.shuffle(bl)
            m, l, o, lse = oracle.online_blocks(s, v, bl)
            assert m == s.max()
            np.testing.assert_allclose(o, o_ref[0], rtol=1e-12, atol=1e-12)
            assert abs(lse - lse_ref[0]) < 1e-12


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_merge_of_random_partition_matches_full(seed):
    rng = np.random.default_rng(200 + seed)
    n, dv = 97, 6
    s = rng.standard_normal(n) * 5
    v = rng.standard_normal((n, dv))
    _, _, o_ref, lse_ref = oracle.online_blocks(s, v, [(0, n)])
    cuts = np.sort(rng.choice(np.arange(1, n), size=6, replace=False))
    edges = [0, *cuts.tolist(), n]
    parts = [(edges[i], edges[i + 1] - edges[i]) for i in range(len(edges) - 1)]
    parts.append((n, 0))  # an empty part must contribute nothing
    ms, ls, os_ = [], [], []
    for (j0, ln) in parts:
        m, l, o, _ = oracle.online_blocks(s, v, [(j0, ln)])
        ms.append(m); ls.append(l); os_.append(o)
    for perm in (list(range(len(parts))), list(range(len(parts)))[::-1], rng.permutation(len(parts)).tolist()):
        m, l, o, lse = oracle.merge([ms[p] for p in perm], [ls[p] for p in perm], [os_[p] for p in perm])
        np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-13)
        assert abs(lse - lse_ref) < 1e-12 and m == s.max()
    # all parts empty -> O = 0, LSE = -inf
    m, l, o, lse = oracle.merge([-math.inf] * 3, [0.0] * 3, np.zeros((3, dv)))
    assert m == -math.inf and l == 0.0 and np.all(o == 0.0) and lse == -math.inf


def test_merge_two_blocks_closed_form():
    # The two-block rule on s = [0 | 5], V = [2 | 3] reproduces practice problem 1.
    e5 = math.exp(-5.0)
    m, l, o, lse = oracle.merge([0.0, 5.0], [1.0, 1.0], [[2.0], [3.0]])
    assert m == 5.0 and abs(l - (1 + e5)) < 1e-15
    assert abs(o[0] - (2 * e5 + 3) / (1 + e5)) < 1e-15


def test_alpha_at_most_one_and_exp_args_nonpositive():
    # The running max never decreases, so every rescale factor is <= 1 and every
    # exponent argument s_j - m is <= 0: the unnormalised l stays <= block count.
    rng = np.random.default_rng(16)
    s = rng.standard_normal(200) * 20
    m, l, _, _ = oracle.online_blocks(s, np.ones(200), [(j, 10) for j in range(0, 200, 10)])
    assert 1.0 <= l <= 200.0 and m == s.max()


# ------------------------------------------------------------ local window

def _window_mask(nq, nk, wl, wr):
    ii = np.arange(nq)[:, None] + (nk - nq)
    jj = np.arange(nk)[None, :]
    vis = np.ones((nq, nk), dtype=bool)
    if wl >= 0:
        vis &= jj >= ii - wl
    if wr >= 0:
        vis &= jj <= ii + wr
    return vis


def test_window_reduces_to_causal_and_full():
    rng = np.random.default_rng(31)
    for nq, nk in ((9, 9), (5, 12), (12, 5)):
        q, k, v = rng.standard_normal((nq, 4)), rng.standard_normal((nk, 4)), rng.standard_normal((nk, 4))
        oc, lc = oracle.attention(q, k, v, 0.7, True)
        ow, lw = oracle.attention_window(q, k, v, 0.7, -1, 0)
        np.testing.assert_array_equal(oc, ow)
        np.testing.assert_array_equal(lc, lw)
        of, lf = oracle.attention(q, k, v, 0.7, False)
        ow, lw = oracle.attention_window(q, k, v, 0.7, -1, -1)
        np.testing.assert_array_equal(of, ow)
        np.testing.assert_array_equal(lf, lw)


@pytest.mark.parametrize("nq,nk,wl,wr,seed", [
    (10, 10, 2, 0, 0), (10, 10, 3, 3, 1), (6, 14, 4, 1, 2), (14, 6, 0, 2, 3), (8, 8, -1, 2, 4), (8, 8, 1, -1, 5),
])
def test_window_matches_scipy_softmax(nq, nk, wl, wr, seed):
    rng = np.random.default_rng(seed)
    d = 3
    q, k, v = rng.standard_normal((nq, d)) * 2, rng.standard_normal((nk, d)), rng.standard_normal((nk, d))
    o, lse = oracle.attention_window(q, k, v, 0.5, wl, wr)
    S = np.where(_window_mask(nq, nk, wl, wr), 0.5 * (q @ k.T), -np.inf)
    for i in range(nq):
        if np.all(np.isneginf(S[i])):
            assert np.all(o[i] == 0.0) and lse[i] == -np.inf
            continue
        np.testing.assert_allclose(o[i], sps.softmax(S[i]) @ v, rtol=1e-12, atol=1e-13)
        assert abs(lse[i] - sps.logsumexp(S[i])) < 1e-12


def test_window_of_one_key_and_uniform_counts():
    rng = np.random.default_rng(32)
    nq, nk, d = 7, 9, 5
    q, k, v = rng.standard_normal((nq, d)), rng.standard_normal((nk, d)), rng.standard_normal((nk, d))
    off = nk - nq
    # window (0, 0): each row sees exactly key i + off
    o, lse = oracle.attention_window(q, k, v, 0.25, 0, 0)
    for i in range(nq):
        np.testing.assert_array_equal(o[i], v[i + off])
        assert abs(lse[i] - 0.25 * (q[i] @ k[i + off])) < 1e-14
    # Q = 0: O is the mean of the visible keys' values, LSE = ln(count)
    o, lse = oracle.attention_window(np.zeros((nq, d)), k, v, 1.0, 2, 1)
    for i in range(nq):
        lo, hi = max(0, i + off - 2), min(nk - 1, i + off + 1)
        np.testing.assert_allclose(o[i], v[lo:hi + 1].mean(axis=0), rtol=1e-13, atol=1e-14)
        assert abs(lse[i] - np.log(hi - lo + 1)) < 1e-14
    # a window entirely past the key axis leaves the row empty
    o, lse = oracle.attention_window(q[:3], k[:2], v[:2], 1.0, 0, 0)  # off = -1: row 0 sees key -1
    assert np.all(o[0] == 0.0) and lse[0] == -np.inf
