"""Standalone row softmax (fa_softmax_rows) against the oracle's two-pass
normaliser ("Online Softmax 算法详解" section 2.2), element by element.

Bound (fp32 arithmetic, exp(x - M) as 2^((x - M) log2 e) with ex2.approx):
the exponent is a rounded difference times a rounded constant, off by about
2^-23 |x - M| log2 e (when one thread's slice is rescaled by exp(m - M) the
two steps' differences add up to the same |x - M|); ex2.approx, the fp32 sums
and the division each add a few ulp.  So
|dy| <= y (4e-6 + 3e-7 |x - M|) + 2^-125, where 2^-125 covers results the
flush-to-zero exponential sends to 0.  bf16 results may also differ by half a
bf16 ulp (their rounding).  |dLSE| <= 1e-5 (1 + |LSE|).
Shapes cover every launch form: one CTA per row at each width, vector and
scalar access, clusters of 2..8 CTAs holding the row on chip or streaming it
twice, and -- with at least two long rows per SM -- one CTA per row streaming
it twice through its ring.
"""
import numpy as np
import pytest
import torch

import oracle
import online_softmax_sm_gb300 as fa
from online_softmax_sm_gb300 import workloads

pytestmark = pytest.mark.gpu


def _bound(x64: np.ndarray, y_ref: np.ndarray, bf16: bool) -> np.ndarray:
    M = np.max(np.where(np.isfinite(x64), x64, -np.inf), axis=1, keepdims=True)
    gap = np.where(np.isfinite(x64) & np.isfinite(M), M - x64, 0.0)
    tol = y_ref * (4e-6 + 3e-7 * gap) + 2.0 ** -125
    if bf16:
        e = np.floor(np.log2(np.where(y_ref > 0, y_ref, 1.0)))
        tol = tol + np.where(y_ref > 0, np.exp2(e - 8), 0.0)
    return tol


def _check(x: torch.Tensor, y: torch.Tensor, lse: torch.Tensor | None, rows=None, what=""):
    x64 = x.detach().cpu().double().numpy()
    if rows is not None:
        x64 = x64[rows]
    y_ref, lse_ref = oracle.softmax_rows(x64)
    yg = y.detach().cpu().double().numpy()
    if rows is not None:
        yg = yg[rows]
    tol = _bound(x64, y_ref, y.dtype == torch.bfloat16)
    err = np.abs(yg - y_ref)
    bad = err > tol
    assert not bad.any(), (f"{what}: {bad.sum()} elements out of bound; worst "
                           f"{(err - tol).max():.3e} at {np.unravel_index(np.argmax(err - tol), err.shape)}")
    if lse is not None:
        lg = lse.detach().cpu().double().numpy()
        if rows is not None:
            lg = lg[rows]
        empty = np.isneginf(lse_ref)
        assert np.all(np.isneginf(lg[empty])), f"{what}: empty rows must give LSE = -inf"
        assert np.all(yg[empty] == 0.0), f"{what}: empty rows must give y = 0"
        d = np.abs(lg[~empty] - lse_ref[~empty])
        assert np.all(d <= 1e-5 * (1 + np.abs(lse_ref[~empty]))), f"{what}: LSE off by {d.max():.3e}"


def _logits(rows, cols, dtype, sigma=4.0, seed=0, specials=True):
    w = workloads.SoftmaxWorkload("t", rows, cols, "f32" if dtype == torch.float32 else "bf16",
                                  sigma=sigma, seed=seed)
    x = workloads.generate_logits(w, device="cuda")
    if specials and rows >= 3:
        x[1, ::3] = float("-inf")          # masked entries
        x[2, :] = float("-inf")            # an empty row
        x[0, :] += 1000.0                  # a large offset: exp against the running max
    return x


# rows, cols: one CTA of 32..1024 threads; scalar access (cols * elt not a
# multiple of 16); clusters of 2, 4, 8; the streaming form.
SHAPES = [(1, 1), (3, 5), (7, 33), (64, 512), (33, 1000), (5, 4097), (9, 16384),
          (4, 16385), (3, 50000), (2, 131072), (3, 131075), (2, 200000), (1, 1 << 20)]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("rows,cols", SHAPES, ids=[f"r{r}c{c}" for r, c in SHAPES])
def test_softmax_rows_all_elements(rows, cols, dtype):
    x = _logits(rows, cols, dtype, seed=rows * 7 + cols)
    y, lse = fa.softmax_rows(x)
    torch.cuda.synchronize()
    _check(x, y, lse, what=f"{rows}x{cols} {dtype}")


# Long rows, at least two per SM: the streaming form, a group of 1, 2, 4 or 8
# CTAs per row by row length, two passes through each CTA's ring of bulk
# copies.  Ragged last sub-chunks (a few columns past a multiple of the
# sub-chunk), chunks of exactly two sub-chunks, and many.
STREAM_SHAPES = [(32776, "bf16"), (16392, "f32"), (65536, "bf16"), (40000, "f32"),
                 (131080, "bf16"), (90000, "f32"), (262152, "bf16"), (131080, "f32")]


@pytest.mark.parametrize("cols,dt", STREAM_SHAPES, ids=[f"c{c}_{d}" for c, d in STREAM_SHAPES])
def test_streaming_rows_all_elements(cols, dt):
    rows = 2 * torch.cuda.get_device_properties(0).multi_processor_count + 5
    dtype = torch.float32 if dt == "f32" else torch.bfloat16
    x = _logits(rows, cols, dtype, seed=rows + cols)
    y, lse = fa.softmax_rows(x)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    _check(x, y, lse, what=f"{rows}x{cols} {dt}")


@pytest.mark.parametrize("cols,dt", [(600008, "f32"), (1200016, "bf16")], ids=["c600008_f32", "c1200016_bf16"])
def test_streaming_very_long_rows_all_elements(cols, dt):
    """Rows long enough for the largest groups: 16 CTAs for fp32 (a
    non-portable cluster size), 8 for bf16; enough rows for every group of
    the grid, every element checked."""
    rows = 40
    dtype = torch.float32 if dt == "f32" else torch.bfloat16
    x = _logits(rows, cols, dtype, seed=cols)
    y, lse = fa.softmax_rows(x)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    _check(x, y, lse, what=f"{rows}x{cols} {dt}")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_in_place_and_without_lse(dtype):
    x = _logits(40, 3000, dtype, seed=5)
    ref = x.clone()
    y_sep, _ = fa.softmax_rows(ref, want_lse=False)
    y, lse = fa.softmax_rows(x, out=x, want_lse=False)
    torch.cuda.synchronize()
    assert lse is None and y.data_ptr() == x.data_ptr()
    assert torch.equal(y, y_sep)
    _check(ref, y, None, what="in place")


def test_rows_sum_to_one_and_repeat_bit_exact():
    """Rows sum to 1 within the per-element bound summed over the row."""
    x = _logits(256, 8192, torch.float32, sigma=8.0, seed=3, specials=False)
    y1, l1 = fa.softmax_rows(x)
    y2, l2 = fa.softmax_rows(x)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2) and torch.equal(l1, l2)
    x64 = x.cpu().double().numpy()
    y_ref, _ = oracle.softmax_rows(x64)
    allowed = _bound(x64, y_ref, False).sum(axis=1)
    s = y1.double().sum(dim=1).cpu().numpy()
    assert np.all(np.abs(s - 1) <= allowed), (np.abs(s - 1) - allowed).max()


@pytest.mark.parametrize("w", list(workloads.SOFTMAX_WORKLOADS.values()), ids=lambda w: w.name)
def test_softmax_workload_sampled(w):
    """The benchmark workloads in their full size and launch form: the first
    and last rows plus seeded samples, every element of those rows."""
    x = workloads.generate_logits(w, device="cuda")
    y, lse = fa.softmax_rows(x)
    torch.cuda.synchronize()
    rng = np.random.default_rng(w.seed)
    rows = sorted({0, w.rows - 1, *rng.integers(0, w.rows, size=6).tolist()})
    _check(x, y, lse, rows=rows, what=w.name)


@pytest.mark.parametrize("rows,cols,dt", [(4, 0, 0), (-1, 8, 0), (4, 8, 7), (4, (1 << 30) + 1, 0)])
def test_bad_arguments_are_rejected(rows, cols, dt):
    x = torch.zeros(64, device="cuda")
    rc = fa.lib().fa_softmax_rows(x.data_ptr(), x.data_ptr(), None, rows, cols, dt, None)
    assert rc == fa.FA_ERR_INVALID_ARG


def test_zero_rows_is_a_no_op():
    x = torch.zeros(4, device="cuda")
    assert fa.lib().fa_softmax_rows(x.data_ptr(), x.data_ptr(), None, 0, 4, 0, None) == fa.FA_OK
