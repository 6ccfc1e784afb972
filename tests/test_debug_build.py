"""The debug build, libfa_debug.so (-DFA_DEBUG).

Its kernels check their runtime indices -- shared-memory ring stages and
staging slots, heads, query rows and key tiles of every TMA copy, global
row indices of O, LSE and the split partials -- and the TMEM column layout
is checked at compile time.  A failed check records FA_ERR_DEVICE_CHECK and
the kernel source line in the device status word and skips the access; no
check traps.  Every shape here must run with all checks passing (status
FA_OK) and still match the fp64 oracle: the small ragged shapes of the parity
tests, the persistent grid with few CTAs, split-KV partials with their merge,
local windows and the E4M3 forward.
"""
import ctypes
import os

import pytest
import torch

import online_softmax_sm_gb300 as fa
from online_softmax_sm_gb300 import _binding, workloads
from online_softmax_sm_gb300 import build as fa_build
from tests import _parity as P
from tests.test_parity import SMALL


@pytest.fixture(scope="module")
def debug_lib():
    fa_build.build(debug=True)  # no-op when up to date
    return _binding.LIB_DEBUG_PATH


def test_debug_library_exports_every_declared_symbol():
    fa_build.build(debug=True)
    L = ctypes.CDLL(_binding.LIB_DEBUG_PATH)
    for name in _binding.declared_symbols():
        assert hasattr(L, name), name


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,n_splits,bc,qt", SMALL,
                         ids=[f"b{c[0]}h{c[1]}q{c[2]}k{c[3]}d{c[4]}{'c' if c[5] else ''}s{c[6]}bc{c[7]}qt{c[8]}"
                              for c in SMALL])
def test_debug_build_small_shapes(debug_lib, B, H, Nq, Nk, d, causal, n_splits, bc, qt):
    w = workloads.custom(B, H, Nq, Nk, d, seed=Nq * 7 + Nk, causal=causal, n_splits=n_splits, bc=bc,
                         q_mult=2.0)
    q, k, v = workloads.generate(w, device="cuda")
    with fa.debug_library():
        assert fa.device_status() == fa.FA_OK
        o, lse = fa.fwd(q, k, v, w.scale, causal, n_splits, bc=bc, q_tiles_per_cta=qt, max_ctas=3)
        torch.cuda.synchronize()
        st = fa.device_status()
        assert st == fa.FA_OK, fa.strerror(st)
    P.compare(q, k, v, o, lse, w.scale, causal).check(w.name + " (debug build)")


@pytest.mark.gpu
def test_debug_build_partials_window_and_fp8(debug_lib):
    w = workloads.custom(2, 3, 300, 700, 128, seed=41, q_mult=2.0)
    q, k, v = workloads.generate(w, device="cuda")
    with fa.debug_library():
        m_p, l_p, o_p = fa.fwd_partial(q, k, v, 3, w.scale, True)
        o_m, lse_m = fa.merge_splits(m_p, l_p, o_p)
        o_w, lse_w = fa.fwd_local(q, k, v, 100, 20, w.scale)
        q8, k8, v8 = (t.to(torch.float8_e4m3fn) for t in (q, k, v))
        o_8, lse_8 = fa.fwd_fp8(q8, k8, v8, w.scale, 1.0, 1.0, 1.0, True)
        torch.cuda.synchronize()
        st = fa.device_status()
        assert st == fa.FA_OK, fa.strerror(st)
    P.compare(q, k, v, o_m, lse_m, w.scale, True).check("partials + merge (debug build)")
    P.compare(q, k, v, o_w, lse_w, w.scale, False, window=(100, 20)).check("window (debug build)")
    # the E4M3 result against the release build's (same kernel code, checks aside)
    o_r, lse_r = fa.fwd_fp8(q8, k8, v8, w.scale, 1.0, 1.0, 1.0, True)
    torch.cuda.synchronize()
    assert torch.equal(o_8, o_r) and torch.equal(lse_8, lse_r)


@pytest.mark.gpu
@pytest.mark.parametrize("rows_per_sm,cols,dt", [(2, 32776, torch.bfloat16), (2, 131080, torch.bfloat16),
                                                  (0, 50000, torch.float32)],
                         ids=["stream_bf16", "stream_group2_bf16", "cluster_f32"])
def test_debug_build_softmax_long_rows(debug_lib, rows_per_sm, cols, dt):
    """The long-row softmax kernels (streaming, one CTA or a group per row,
    and the ring kernel's cluster for few rows) under the debug build's
    bounds checks, bit-equal to release."""
    rows = max(3, rows_per_sm * torch.cuda.get_device_properties(0).multi_processor_count + 3)
    x = (torch.randn(rows, cols, device="cuda", generator=torch.Generator("cuda").manual_seed(cols))
         * 4.0).to(dt)
    with fa.debug_library():
        y_d, lse_d = fa.softmax_rows(x)
        torch.cuda.synchronize()
        st = fa.device_status()
        assert st == fa.FA_OK, fa.strerror(st)
    y_r, lse_r = fa.softmax_rows(x)
    torch.cuda.synchronize()
    assert torch.equal(y_d, y_r) and torch.equal(lse_d, lse_r)
