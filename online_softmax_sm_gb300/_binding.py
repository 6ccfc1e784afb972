"""ctypes binding of libfa.so (include/fa.h).

Argument marshalling only: every step of the attention forward runs in the
library's CUDA kernels.  torch supplies device memory and the current stream.
If libfa.so is missing, every call raises: there is no fallback path.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import re

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfa.so")
LIB_DEBUG_PATH = os.path.join(PKG, "libfa_debug.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "fa.h")

FA_OK = 0
FA_ERR_INVALID_ARG = -1
FA_ERR_UNSUPPORTED = -2
FA_ERR_CUDA = -3
FA_ERR_DEVICE_TIMEOUT = -4
FA_ERR_NO_MEMORY = -5
FA_ERR_SCRATCH_TOO_SMALL = -6
FA_ERR_DEVICE_CHECK = -7
FA_DTYPE_F32 = 0
FA_DTYPE_BF16 = 1
NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


class FaOpts(ctypes.Structure):
    _fields_ = [("bc", ctypes.c_int), ("q_tiles_per_cta", ctypes.c_int),
                ("timeout_ns", ctypes.c_ulonglong), ("test_skip_kv_load", ctypes.c_int),
                ("max_ctas", ctypes.c_int)]


class FAError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {strerror(code)} (code {code})")
        self.code = code


_lib = None
_vp = ctypes.c_void_p
_fp = ctypes.POINTER(ctypes.c_float)
_i = ctypes.c_int


def _declare(L):
    L.fa_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, ctypes.c_float, _i, _i, _vp]
    L.fa_fwd.restype = _i
    L.fa_fwd_ex.argtypes = L.fa_fwd.argtypes + [ctypes.POINTER(FaOpts)]
    L.fa_fwd_ex.restype = _i
    L.fa_fwd_partial.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, ctypes.c_float,
                                 _i, _i, _vp]
    L.fa_fwd_partial.restype = _i
    L.fa_merge_splits.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp]
    L.fa_merge_splits.restype = _i
    L.fa_split_workspace_bytes.argtypes = [_i, _i, _i, _i, _i]
    L.fa_split_workspace_bytes.restype = ctypes.c_size_t
    L.fa_get_device_status.argtypes = [_vp]
    L.fa_get_device_status.restype = _i
    L.fa_strerror.argtypes = [_i]
    L.fa_strerror.restype = ctypes.c_char_p
    L.fa_version.argtypes = []
    L.fa_version.restype = _i
    L.fa_fwd_split_noalloc.argtypes = L.fa_fwd.argtypes
    L.fa_fwd_split_noalloc.restype = _i
    L.fa_fwd_local.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, ctypes.c_float, _i, _i,
                               _i, _vp]
    L.fa_fwd_local.restype = _i
    L.fa_fwd_host.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, ctypes.c_float, _i, _i]
    L.fa_fwd_host.restype = _i
    L.fa_fwd_local_host.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, ctypes.c_float, _i, _i, _i]
    L.fa_fwd_local_host.restype = _i
    L.fa_fwd_fp8_host.argtypes = [_vp] * 5 + [_i] * 5 + [ctypes.c_float] * 4 + [_i, _i]
    L.fa_fwd_fp8_host.restype = _i
    L.fa_softmax_rows.argtypes = [_vp, _vp, _vp, ctypes.c_longlong, _i, _i, _vp]
    L.fa_softmax_rows.restype = _i
    L.fa_fwd_fp8.argtypes = [_vp] * 5 + [_i] * 5 + [ctypes.c_float] * 4 + [_i, _vp]
    L.fa_fwd_fp8.restype = _i
    L.fa_bwd.argtypes = [_vp] * 9 + [_i] * 5 + [ctypes.c_float, _i, _vp]
    L.fa_bwd.restype = _i
    L.fa_bwd_local.argtypes = [_vp] * 9 + [_i] * 5 + [ctypes.c_float, _i, _i, _vp]
    L.fa_bwd_local.restype = _i
    L.fa_bwd_host.argtypes = [_vp] * 9 + [_i] * 5 + [ctypes.c_float, _i, _i]
    L.fa_bwd_host.restype = _i
    L.fa_bwd_local_host.argtypes = [_vp] * 9 + [_i] * 5 + [ctypes.c_float, _i, _i, _i]
    L.fa_bwd_local_host.restype = _i


def lib():
    """The loaded libfa.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is not built; run `python -m online_softmax_sm_gb300.build` "
                "(or __graft_entry__.build()).  There is no fallback implementation.")
        L = ctypes.CDLL(LIB_PATH)
        _declare(L)
        _lib = L
    return _lib


@contextlib.contextmanager
def debug_library():
    """Within the block every call goes through libfa_debug.so, the FA_DEBUG
    build: device-side index, shared-memory and TMEM range checks that record
    FA_ERR_DEVICE_CHECK (with the kernel source line, see strerror) in the
    status word and skip the access instead of trapping."""
    global _lib
    if not os.path.exists(LIB_DEBUG_PATH):
        raise RuntimeError(f"{LIB_DEBUG_PATH} is not built; run `python -m online_softmax_sm_gb300.build --debug`")
    L = ctypes.CDLL(LIB_DEBUG_PATH)
    _declare(L)
    saved, _lib = _lib, L
    try:
        yield L
    finally:
        _lib = saved


def declared_symbols(header: str = HEADER) -> list[str]:
    """Function names declared in include/fa.h."""
    with open(header, encoding="utf-8") as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(fa_\w+)\s*\(", text, re.M)))


def strerror(code: int) -> str:
    return lib().fa_strerror(int(code)).decode()


def _check(rc: int, what: str):
    if rc != FA_OK:
        raise FAError(rc, what)


def _stream_handle(dev: torch.device, stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    return s.cuda_stream


def _check_qkv(q, k, v):
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.dtype != torch.bfloat16:
            raise ValueError(f"{name} must be bfloat16")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [B, H, N, d] tensor")
    B, H, Nq, d = q.shape
    if k.shape[:2] != (B, H) or k.shape[3] != d or v.shape != k.shape:
        raise ValueError("k and v must be [B, H, Nk, d] matching q")
    if not (q.device == k.device == v.device):
        raise ValueError("q, k, v must be on one device")
    return B, H, Nq, k.shape[2], d


def fwd(q, k, v, scale: float | None = None, causal: bool = False, n_splits: int = 1,
        out=None, lse=None, bc: int = 0, q_tiles_per_cta: int = 0, timeout_ns: int = 0,
        test_skip_kv_load: int = 0, max_ctas: int = 0, stream=None):
    """fa_fwd / fa_fwd_ex.  Returns (o bf16 [B,H,Nq,d], lse fp32 [B,H,Nq])."""
    B, H, Nq, Nk, d = _check_qkv(q, k, v)
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    assert out.shape == q.shape and out.dtype == torch.bfloat16 and out.is_contiguous()
    assert lse.shape == (B, H, Nq) and lse.dtype == torch.float32 and lse.is_contiguous()
    L = lib()
    with torch.cuda.device(q.device):
        sh = _stream_handle(q.device, stream)
        args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                B, H, Nq, Nk, d, float(scale), int(bool(causal)), int(n_splits), sh)
        if bc or q_tiles_per_cta or timeout_ns or test_skip_kv_load or max_ctas:
            opts = FaOpts(int(bc), int(q_tiles_per_cta), int(timeout_ns), int(test_skip_kv_load),
                          int(max_ctas))
            rc = L.fa_fwd_ex(*args, ctypes.byref(opts))
        else:
            rc = L.fa_fwd(*args)
    _check(rc, "fa_fwd")
    return out, lse


def fwd_host(q, k, v, scale: float | None = None, causal: bool = False, out=None, lse=None,
             n_chunks: int = 0, device=None, window=None):
    """fa_fwd_host: q, k, v are CPU bf16 [B, H, N, d] tensors (page-locked for overlap); the
    call copies them to the device, runs the forward there and copies O and LSE back into
    CPU tensors.  Returns (o bf16 [B,H,Nq,d], lse fp32 [B,H,Nq]) on the CPU.
    window=(window_left, window_right) selects fa_fwd_local_host (the mask of fwd_local)."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or t.device.type != "cpu":
            raise ValueError(f"{name} must be a CPU tensor")
        if t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bfloat16 [B, H, N, d] tensor")
    B, H, Nq, d = q.shape
    if k.shape[:2] != (B, H) or k.shape[3] != d or v.shape != k.shape:
        raise ValueError("k and v must be [B, H, Nk, d] matching q")
    Nk = k.shape[2]
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=q.is_pinned())
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, pin_memory=q.is_pinned())
    if out.device.type != "cpu" or out.shape != q.shape or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous CPU bfloat16 tensor shaped like q")
    if lse.device.type != "cpu" or lse.shape != (B, H, Nq) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous CPU float32 [B, H, Nq] tensor")
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        if window is None:
            rc = lib().fa_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                   B, H, Nq, Nk, d, float(scale), int(bool(causal)), int(n_chunks))
        else:
            rc = lib().fa_fwd_local_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                         lse.data_ptr(), B, H, Nq, Nk, d, float(scale), int(window[0]),
                                         int(window[1]), int(n_chunks))
    _check(rc, "fa_fwd_host" if window is None else "fa_fwd_local_host")
    return out, lse


def fwd_local(q, k, v, window_left: int, window_right: int, scale: float | None = None,
              n_splits: int = 1, out=None, lse=None, stream=None):
    """fa_fwd_local: key j visible to query i iff
    i + (Nk - Nq) - window_left <= j <= i + (Nk - Nq) + window_right (-1 = open side)."""
    B, H, Nq, Nk, d = _check_qkv(q, k, v)
    if scale is None:
        scale = d ** -0.5
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device) if lse is None else lse
    with torch.cuda.device(q.device):
        rc = lib().fa_fwd_local(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                lse.data_ptr(), B, H, Nq, Nk, d, float(scale), int(window_left),
                                int(window_right), int(n_splits), _stream_handle(q.device, stream))
    _check(rc, "fa_fwd_local")
    return out, lse


def fwd_fp8(q8, k8, v8, scale: float | None = None, q_descale: float = 1.0, k_descale: float = 1.0,
            v_descale: float = 1.0, causal: bool = False, out=None, lse=None, stream=None):
    """fa_fwd_fp8: q8, k8, v8 float8_e4m3fn [B, H, N, 128].  Returns (o bf16, lse fp32)."""
    for name, t in (("q8", q8), ("k8", k8), ("v8", v8)):
        if not isinstance(t, torch.Tensor) or t.device.type != "cuda" or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
        if t.dtype != torch.float8_e4m3fn:
            raise ValueError(f"{name} must be float8_e4m3fn")
    B, H, Nq, d = q8.shape
    Nk = k8.shape[2]
    if k8.shape != (B, H, Nk, d) or v8.shape != k8.shape:
        raise ValueError("k8 and v8 must be [B, H, Nk, d] matching q8")
    if scale is None:
        scale = d ** -0.5
    out = torch.empty((B, H, Nq, d), dtype=torch.bfloat16, device=q8.device) if out is None else out
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q8.device) if lse is None else lse
    with torch.cuda.device(q8.device):
        rc = lib().fa_fwd_fp8(q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), out.data_ptr(), lse.data_ptr(),
                              B, H, Nq, Nk, d, float(scale), float(q_descale), float(k_descale),
                              float(v_descale), int(bool(causal)), _stream_handle(q8.device, stream))
    _check(rc, "fa_fwd_fp8")
    return out, lse


def fwd_fp8_host(q8, k8, v8, scale: float | None = None, q_descale: float = 1.0, k_descale: float = 1.0,
                 v_descale: float = 1.0, causal: bool = False, out=None, lse=None, n_chunks: int = 0,
                 device=None):
    """fa_fwd_fp8_host: q8, k8, v8 CPU float8_e4m3fn [B, H, N, 128] tensors (page-locked for
    overlap); copies in, the FP8 forward, O (bf16) and LSE (fp32) back into CPU tensors."""
    for name, t in (("q8", q8), ("k8", k8), ("v8", v8)):
        if not isinstance(t, torch.Tensor) or t.device.type != "cpu" or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CPU tensor")
        if t.dtype != torch.float8_e4m3fn or t.dim() != 4:
            raise ValueError(f"{name} must be a float8_e4m3fn [B, H, N, d] tensor")
    B, H, Nq, d = q8.shape
    Nk = k8.shape[2]
    if k8.shape != (B, H, Nk, d) or v8.shape != k8.shape:
        raise ValueError("k8 and v8 must be [B, H, Nk, d] matching q8")
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty((B, H, Nq, d), dtype=torch.bfloat16, pin_memory=q8.is_pinned())
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, pin_memory=q8.is_pinned())
    if out.device.type != "cpu" or out.shape != (B, H, Nq, d) or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous CPU bfloat16 [B, H, Nq, d] tensor")
    if lse.device.type != "cpu" or lse.shape != (B, H, Nq) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous CPU float32 [B, H, Nq] tensor")
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        rc = lib().fa_fwd_fp8_host(q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), out.data_ptr(),
                                   lse.data_ptr(), B, H, Nq, Nk, d, float(scale), float(q_descale),
                                   float(k_descale), float(v_descale), int(bool(causal)), int(n_chunks))
    _check(rc, "fa_fwd_fp8_host")
    return out, lse


def bwd(q, k, v, o, lse, dout, scale: float | None = None, causal: bool = False, window=None,
        dq=None, dk=None, dv=None, stream=None):
    """fa_bwd / fa_bwd_local: (dq, dk, dv) bf16, shapes of q, k, v.  `o` and
    `lse` are the forward's outputs; window=(wl, wr) selects fa_bwd_local."""
    B, H, Nq, Nk, d = _check_qkv(q, k, v)
    for name, t in (("o", o), ("dout", dout)):
        if t.shape != q.shape or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 tensor shaped like q")
    if lse.shape != (B, H, Nq) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B, H, Nq] tensor")
    if scale is None:
        scale = d ** -0.5
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    args = [q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dout.data_ptr(),
            dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Nq, Nk, d, float(scale)]
    with torch.cuda.device(q.device):
        sh = _stream_handle(q.device, stream)
        if window is None:
            rc = lib().fa_bwd(*args, int(bool(causal)), sh)
        else:
            rc = lib().fa_bwd_local(*args, int(window[0]), int(window[1]), sh)
    _check(rc, "fa_bwd")
    return dq, dk, dv


def bwd_host(q, k, v, o, lse, dout, scale: float | None = None, causal: bool = False, window=None,
             dq=None, dk=None, dv=None, n_chunks: int = 0, device=None):
    """fa_bwd_host / fa_bwd_local_host: every tensor on the CPU (page-locked for overlap); the
    call copies the inputs to the device, runs the backward and copies dq, dk, dv back."""
    ts = {"q": q, "k": k, "v": v, "o": o, "dout": dout}
    for name, t in ts.items():
        if not isinstance(t, torch.Tensor) or t.device.type != "cpu" or t.dtype != torch.bfloat16 \
                or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CPU bfloat16 [B, H, N, d] tensor")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if k.shape != (B, H, Nk, d) or v.shape != k.shape or o.shape != q.shape or dout.shape != q.shape:
        raise ValueError("shapes: q, o, dout [B, H, Nq, d]; k, v [B, H, Nk, d]")
    if (not isinstance(lse, torch.Tensor) or lse.device.type != "cpu" or lse.shape != (B, H, Nq)
            or lse.dtype != torch.float32 or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous CPU float32 [B, H, Nq] tensor")
    if scale is None:
        scale = d ** -0.5
    pin = q.is_pinned()
    dq = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=pin) if dq is None else dq
    dk = torch.empty(k.shape, dtype=torch.bfloat16, pin_memory=pin) if dk is None else dk
    dv = torch.empty(v.shape, dtype=torch.bfloat16, pin_memory=pin) if dv is None else dv
    for name, t, ref in (("dq", dq, q), ("dk", dk, k), ("dv", dv, v)):
        if t.device.type != "cpu" or t.shape != ref.shape or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CPU bfloat16 tensor shaped like its input")
    args = [q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dout.data_ptr(),
            dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Nq, Nk, d, float(scale)]
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        if window is None:
            rc = lib().fa_bwd_host(*args, int(bool(causal)), int(n_chunks))
        else:
            rc = lib().fa_bwd_local_host(*args, int(window[0]), int(window[1]), int(n_chunks))
    _check(rc, "fa_bwd_host")
    return dq, dk, dv


def fwd_partial(q, k, v, n_splits: int, scale: float | None = None, causal: bool = False,
                m_part=None, l_part=None, o_part=None, stream=None):
    """fa_fwd_partial.  Returns (m_part [S,B,H,Nq], l_part [S,B,H,Nq], o_part [S,B,H,Nq,d])."""
    B, H, Nq, Nk, d = _check_qkv(q, k, v)
    if scale is None:
        scale = d ** -0.5
    dev = q.device
    f32 = dict(dtype=torch.float32, device=dev)
    m_part = torch.empty((n_splits, B, H, Nq), **f32) if m_part is None else m_part
    l_part = torch.empty((n_splits, B, H, Nq), **f32) if l_part is None else l_part
    o_part = torch.empty((n_splits, B, H, Nq, d), **f32) if o_part is None else o_part
    L = lib()
    with torch.cuda.device(dev):
        rc = L.fa_fwd_partial(q.data_ptr(), k.data_ptr(), v.data_ptr(), m_part.data_ptr(),
                              l_part.data_ptr(), o_part.data_ptr(), B, H, Nq, Nk, d, float(scale),
                              int(bool(causal)), int(n_splits), _stream_handle(dev, stream))
    _check(rc, "fa_fwd_partial")
    return m_part, l_part, o_part


def merge_splits(m_part, l_part, o_part, out=None, lse=None, stream=None):
    """fa_merge_splits.  Returns (o bf16 [B,H,Nq,d], lse fp32 [B,H,Nq])."""
    S, B, H, Nq, d = o_part.shape
    for t in (m_part, l_part, o_part):
        if t.dtype != torch.float32 or not t.is_contiguous() or t.device.type != "cuda":
            raise ValueError("partials must be contiguous fp32 CUDA tensors")
    assert m_part.shape == (S, B, H, Nq) and l_part.shape == (S, B, H, Nq)
    dev = o_part.device
    out = torch.empty((B, H, Nq, d), dtype=torch.bfloat16, device=dev) if out is None else out
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=dev) if lse is None else lse
    L = lib()
    with torch.cuda.device(dev):
        rc = L.fa_merge_splits(m_part.data_ptr(), l_part.data_ptr(), o_part.data_ptr(),
                               out.data_ptr(), lse.data_ptr(), B, H, Nq, d, S,
                               _stream_handle(dev, stream))
    _check(rc, "fa_merge_splits")
    return out, lse


def fwd_split_noalloc(q, k, v, n_splits: int, scale: float | None = None, causal: bool = False,
                      out=None, lse=None, stream=None):
    """fa_fwd_split_noalloc: split-KV forward whose workspace is the library's
    fixed device scratch (no allocation on the call path).  Calls that may
    overlap on the GPU share that scratch and must be serialised by the caller."""
    B, H, Nq, Nk, d = _check_qkv(q, k, v)
    if scale is None:
        scale = d ** -0.5
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device) if lse is None else lse
    with torch.cuda.device(q.device):
        rc = lib().fa_fwd_split_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                        lse.data_ptr(), B, H, Nq, Nk, d, float(scale),
                                        int(bool(causal)), int(n_splits),
                                        _stream_handle(q.device, stream))
    _check(rc, "fa_fwd_split_noalloc")
    return out, lse


def softmax_rows(x, out=None, lse=None, want_lse: bool = True, stream=None):
    """fa_softmax_rows over the last dimension of x (fp32 or bf16, contiguous).
    Returns (y, lse) with lse fp32 of shape x.shape[:-1], or (y, None)."""
    if not isinstance(x, torch.Tensor) or x.device.type != "cuda" or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA tensor")
    if x.dtype == torch.float32:
        dt = FA_DTYPE_F32
    elif x.dtype == torch.bfloat16:
        dt = FA_DTYPE_BF16
    else:
        raise ValueError("x must be float32 or bfloat16")
    if x.dim() < 1 or x.shape[-1] < 1:
        raise ValueError("x needs a non-empty last dimension")
    cols = x.shape[-1]
    rows = x.numel() // cols
    out = torch.empty_like(x) if out is None else out
    assert out.shape == x.shape and out.dtype == x.dtype and out.is_contiguous()
    if want_lse and lse is None:
        lse = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    with torch.cuda.device(x.device):
        rc = lib().fa_softmax_rows(x.data_ptr(), out.data_ptr(),
                                   lse.data_ptr() if lse is not None else None, rows, cols, dt,
                                   _stream_handle(x.device, stream))
    _check(rc, "fa_softmax_rows")
    return out, lse


def split_workspace_bytes(B: int, H: int, Nq: int, d: int, n_splits: int) -> int:
    return int(lib().fa_split_workspace_bytes(B, H, Nq, d, n_splits))


def device_status(device=None, stream=None) -> int:
    """fa_get_device_status on `device` (default: current).  Returns the FA_* code."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        return int(lib().fa_get_device_status(_stream_handle(dev, stream)))


def version() -> int:
    return int(lib().fa_version())
