"""C-ABI checks that need no GPU: libfa.so loads, exports every function
include/fa.h declares, and rejects bad arguments before launching anything."""
import ctypes
import os

import pytest

import online_softmax_sm_gb300 as fa
from online_softmax_sm_gb300 import _binding, build


@pytest.fixture(scope="module")
def L():
    build.build()  # no-op when up to date (nvcc cross-compiles without a GPU)
    return fa.lib()


def test_exports_every_declared_symbol(L):
    names = _binding.declared_symbols()
    assert {"fa_fwd", "fa_merge_splits", "fa_fwd_partial", "fa_fwd_ex", "fa_get_device_status",
            "fa_strerror", "fa_split_workspace_bytes", "fa_version"} <= set(names)
    raw = ctypes.CDLL(_binding.LIB_PATH)
    for name in names:
        assert hasattr(raw, name), f"libfa.so does not export {name}"


def test_version_and_strerror(L):
    assert fa.version() == 101
    for code in (fa.FA_OK, fa.FA_ERR_INVALID_ARG, fa.FA_ERR_UNSUPPORTED, fa.FA_ERR_CUDA,
                 fa.FA_ERR_DEVICE_TIMEOUT, fa.FA_ERR_NO_MEMORY, -99):
        s = fa.strerror(code)
        assert isinstance(s, str) and s


def test_split_workspace_bytes(L):
    assert fa.split_workspace_bytes(1, 1, 128, 128, 1) == 0
    assert fa.split_workspace_bytes(1, 1, 128, 96, 4) == 0
    n = fa.split_workspace_bytes(16, 32, 128, 128, 16)
    rows = 16 * 32 * 128
    # m and l fp32, O bf16 (fa_fwd's own split workspace)
    assert n >= 16 * rows * (2 * 4 + 128 * 2) and n % 256 == 0


def _fwd(L, q=0x1000, k=0x1000, v=0x1000, o=0x1000, lse=0x1000, B=1, H=1, Nq=8, Nk=8, d=64,
         scale=0.125, causal=0, n_splits=1):
    return L.fa_fwd(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, n_splits, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), fa.FA_ERR_INVALID_ARG),
    (dict(o=None), fa.FA_ERR_INVALID_ARG),
    (dict(lse=None), fa.FA_ERR_INVALID_ARG),
    (dict(q=0x1008), fa.FA_ERR_INVALID_ARG),       # not 16-byte aligned
    (dict(lse=0x1002), fa.FA_ERR_INVALID_ARG),     # not 4-byte aligned
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(Nq=0), fa.FA_ERR_INVALID_ARG),
    (dict(Nk=-5), fa.FA_ERR_INVALID_ARG),
    (dict(Nq=(1 << 30) + 1), fa.FA_ERR_INVALID_ARG),
    (dict(B=256, H=256), fa.FA_ERR_INVALID_ARG),   # B*H > 65535
    (dict(scale=0.0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=-1.0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(n_splits=0), fa.FA_ERR_INVALID_ARG),
    (dict(n_splits=70000), fa.FA_ERR_INVALID_ARG),
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(d=256), fa.FA_ERR_UNSUPPORTED),
])
def test_invalid_arguments_rejected_before_launch(L, kw, code):
    assert _fwd(L, **kw) == code


def test_invalid_options_and_partial_and_merge_args(L):
    opts = _binding.FaOpts(96, 0, 0, 0)
    assert L.fa_fwd_ex(0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 1, 1, 8, 8, 64, 0.125, 0, 1, None,
                       ctypes.byref(opts)) == fa.FA_ERR_INVALID_ARG
    opts = _binding.FaOpts(0, 3, 0, 0)
    assert L.fa_fwd_ex(0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 1, 1, 8, 8, 64, 0.125, 0, 1, None,
                       ctypes.byref(opts)) == fa.FA_ERR_INVALID_ARG
    # fa_fwd_partial: o_part must be 16-byte aligned; m_part non-null
    assert L.fa_fwd_partial(0x1000, 0x1000, 0x1000, None, 0x1000, 0x1000, 1, 1, 8, 8, 64, 0.125, 0,
                            2, None) == fa.FA_ERR_INVALID_ARG
    assert L.fa_fwd_partial(0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0x1004, 1, 1, 8, 8, 64, 0.125,
                            0, 2, None) == fa.FA_ERR_INVALID_ARG
    # fa_merge_splits argument checks
    assert L.fa_merge_splits(None, 0x1000, 0x1000, 0x1000, 0x1000, 1, 1, 8, 64, 2, None) == fa.FA_ERR_INVALID_ARG
    assert L.fa_merge_splits(0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 1, 1, 8, 80, 2, None) == fa.FA_ERR_UNSUPPORTED
    assert L.fa_merge_splits(0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 1, 1, 8, 64, 0, None) == fa.FA_ERR_INVALID_ARG
    assert L.fa_merge_splits(0x1000, 0x1000, 0x1008, 0x1000, 0x1000, 1, 1, 8, 64, 2, None) == fa.FA_ERR_INVALID_ARG
    # fa_fwd_host: sizes and null pointers checked before any device work
    assert L.fa_fwd_host(None, 0x1000, 0x1000, 0x1000, 0x1000, 1, 1, 8, 8, 64, 0.125, 0, 0) == fa.FA_ERR_INVALID_ARG
    assert L.fa_fwd_host(0x1000, 0x1000, 0x1000, 0x1000, None, 1, 1, 8, 8, 64, 0.125, 0, 0) == fa.FA_ERR_INVALID_ARG
    assert L.fa_fwd_host(0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0, 1, 8, 8, 64, 0.125, 0, 0) == fa.FA_ERR_INVALID_ARG
    assert L.fa_fwd_host(0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 1, 1, 8, 8, 96, 0.125, 0, 0) == fa.FA_ERR_UNSUPPORTED
    # fa_fwd_local_host: also the window bounds
    assert L.fa_fwd_local_host(None, 0x1000, 0x1000, 0x1000, 0x1000, 1, 1, 8, 8, 64, 0.125, 4, 0, 0) == fa.FA_ERR_INVALID_ARG
    assert L.fa_fwd_local_host(0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 1, 1, 8, 8, 64, 0.125, -2, 0, 0) == fa.FA_ERR_INVALID_ARG
    assert L.fa_fwd_local_host(0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 1, 1, 8, 8, 64, 0.125, 4, (1 << 30) + 1, 0) == fa.FA_ERR_INVALID_ARG
    # fa_fwd_fp8_host: d = 128 only, descales finite and > 0
    assert L.fa_fwd_fp8_host(0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 1, 1, 8, 8, 64, 0.125, 1.0, 1.0, 1.0, 0, 0) == fa.FA_ERR_UNSUPPORTED
    assert L.fa_fwd_fp8_host(0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 1, 1, 8, 8, 128, 0.125, 0.0, 1.0, 1.0, 0, 0) == fa.FA_ERR_INVALID_ARG
    assert L.fa_fwd_fp8_host(None, 0x1000, 0x1000, 0x1000, 0x1000, 1, 1, 8, 8, 128, 0.125, 1.0, 1.0, 1.0, 0, 0) == fa.FA_ERR_INVALID_ARG
    # fa_bwd_host / fa_bwd_local_host: null pointers, sizes, window bounds
    P9 = [0x1000] * 9
    assert L.fa_bwd_host(*([None] + P9[1:]), 1, 1, 8, 8, 64, 0.125, 0, 0) == fa.FA_ERR_INVALID_ARG
    assert L.fa_bwd_host(*P9, 1, 1, 8, 8, 96, 0.125, 0, 0) == fa.FA_ERR_UNSUPPORTED
    assert L.fa_bwd_local_host(*P9, 1, 1, 8, 8, 64, 0.125, -3, 0, 0) == fa.FA_ERR_INVALID_ARG


def test_product_path_fails_loudly_without_library(tmp_path, monkeypatch):
    monkeypatch.setattr(_binding, "LIB_PATH", str(tmp_path / "missing" / "libfa.so"))
    monkeypatch.setattr(_binding, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        _binding.lib()


def test_package_holds_no_oracle_import():
    # The product package must never route through the CPU oracle.
    pkg = os.path.dirname(fa.__file__)
    for root, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                with open(os.path.join(root, fn), encoding="utf-8") as f:
                    text = f.read()
                assert "import oracle" not in text and "from oracle" not in text, fn
