"""fp64 CPU oracle for the online-softmax attention forward.

TEST INFRASTRUCTURE.  Only `tests/`, `__graft_entry__.smoke()` and the
benchmark's `cpu_baseline` / reference leg may import this package.  It never
imports the GPU package and shares no code with it; both sides only share the
seeded input generators, which hold none of the method's arithmetic.

The arithmetic lives in oracle.c (plain C, fp64); this module is ctypes
marshalling plus per-head looping:

  attention(q, k, v, scale, causal, rows)     one head, three-pass definition
  attention_window(q, k, v, scale, wl, wr)     one head, local (sliding-window) mask
  attention_bhnd(q, k, v, scale, causal, ...) [B,H,N,d] tensors, head by head
  online_blocks(s, v, blocks)                 blockwise (m, l, O) recurrence
  merge(m, l, o)                              two-block merge rule, folded
  softmax_two_pass(x)                         Milakov & Gimelshein normaliser

Inputs are upcast exactly to fp64 before the call (bf16 -> fp64 is exact).
"""
from __future__ import annotations

import ctypes
import os
from typing import Iterable, Sequence

import numpy as np

from . import build as _build

_lib = None
_i64 = ctypes.c_int64
_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int64)


def load(path: str | None = None):
    """Load (building first if needed) the oracle library."""
    global _lib
    if path is not None:
        lib = ctypes.CDLL(path)
        _declare(lib)
        return lib
    if _lib is None:
        _lib = ctypes.CDLL(_build.build())
        _declare(_lib)
    return _lib


def _declare(lib):
    lib.oracle_attention.argtypes = [_dp, _i64, _dp, _dp, _i64, _i64, ctypes.c_double,
                                     ctypes.c_int, _ip, _i64, _dp, _dp, ctypes.c_int]
    lib.oracle_attention.restype = ctypes.c_int
    lib.oracle_attention_window.argtypes = [_dp, _i64, _dp, _dp, _i64, _i64, ctypes.c_double,
                                            _i64, _i64, _ip, _i64, _dp, _dp, ctypes.c_int]
    lib.oracle_attention_window.restype = ctypes.c_int
    lib.oracle_online_blocks.argtypes = [_dp, _dp, _i64, _i64, _ip, _ip, _i64,
                                         _dp, _dp, _dp, _dp]
    lib.oracle_online_blocks.restype = ctypes.c_int
    lib.oracle_merge.argtypes = [_dp, _dp, _dp, _i64, _i64, _dp, _dp, _dp, _dp]
    lib.oracle_merge.restype = ctypes.c_int
    lib.oracle_softmax_two_pass.argtypes = [_dp, _i64, _dp, _dp]
    lib.oracle_softmax_two_pass.restype = ctypes.c_int
    lib.oracle_softmax_rows.argtypes = [_dp, _i64, _i64, _ip, _i64, _dp, _dp, ctypes.c_int]
    lib.oracle_softmax_rows.restype = ctypes.c_int
    lib.oracle_attention_bwd.argtypes = [_dp, _i64, _dp, _dp, _i64, _i64, ctypes.c_double, _i64,
                                         _i64, _dp, _dp, _dp, _dp, _dp, _dp, ctypes.c_int]
    lib.oracle_attention_bwd.restype = ctypes.c_int
    lib.oracle_e4m3.argtypes = [ctypes.c_double]
    lib.oracle_e4m3.restype = ctypes.c_double
    lib.oracle_attention_fp8.argtypes = [_dp, _i64, _dp, _dp, _i64, _i64, ctypes.c_double,
                                         ctypes.c_double, ctypes.c_double, ctypes.c_double,
                                         ctypes.c_int, _i64, _ip, _i64, _dp, _dp]
    lib.oracle_attention_fp8.restype = ctypes.c_int


def _f64(a) -> np.ndarray:
    """Exact upcast of a numpy array or a (CPU) torch tensor to C-contiguous fp64."""
    if hasattr(a, "detach"):
        # torch tensor (bf16/fp16/fp32): .double() is exact for these types
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray, t=_dp):
    return a.ctypes.data_as(t)


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


def attention(q, k, v, scale: float, causal: bool = False, rows: Sequence[int] | None = None,
              threads: int | None = None, lib=None):
    """One head: q [nq,d], k [nk,d], v [nk,d].  Returns (o [len(rows),d], lse [len(rows)])."""
    lib = lib or load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    nq, d = q.shape
    nk = k.shape[0]
    assert k.shape == (nk, d) and v.shape == (nk, d)
    if rows is None:
        rows_arr = None
        nrows = nq
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = rows_arr.shape[0]
    o = np.empty((nrows, d), dtype=np.float64)
    lse = np.empty((nrows,), dtype=np.float64)
    rc = lib.oracle_attention(_ptr(q), nq, _ptr(k), _ptr(v), nk, d, float(scale), int(bool(causal)),
                              None if rows_arr is None else _ptr(rows_arr, _ip), nrows,
                              _ptr(o), _ptr(lse), int(threads or default_threads()))
    if rc != 0:
        raise ValueError("oracle_attention: bad argument")
    return o, lse


def attention_window(q, k, v, scale: float, window_left: int, window_right: int,
                     rows: Sequence[int] | None = None, threads: int | None = None, lib=None):
    """One head with the local window: key j visible to query i iff
    i + (nk - nq) - window_left <= j <= i + (nk - nq) + window_right (a negative
    bound leaves that side open).  Returns (o, lse) like attention()."""
    lib = lib or load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    nq, d = q.shape
    nk = k.shape[0]
    assert k.shape == (nk, d) and v.shape == (nk, d)
    if rows is None:
        rows_arr, nrows = None, nq
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = rows_arr.shape[0]
    o = np.empty((nrows, d), dtype=np.float64)
    lse = np.empty((nrows,), dtype=np.float64)
    rc = lib.oracle_attention_window(_ptr(q), nq, _ptr(k), _ptr(v), nk, d, float(scale),
                                     int(window_left), int(window_right),
                                     None if rows_arr is None else _ptr(rows_arr, _ip), nrows,
                                     _ptr(o), _ptr(lse), int(threads or default_threads()))
    if rc != 0:
        raise ValueError("oracle_attention_window: bad argument")
    return o, lse


def attention_bhnd(q, k, v, scale: float, causal: bool = False,
                   heads: Iterable[tuple[int, int]] | None = None,
                   rows: Sequence[int] | None = None, threads: int | None = None, lib=None):
    """q [B,H,Nq,d], k/v [B,H,Nk,d] (numpy or torch).  For each (b,h) in `heads`
    (default: all) computes the listed `rows` (default: all).
    Returns dict {(b,h): (o, lse)}."""
    B, H = q.shape[0], q.shape[1]
    heads = list(heads) if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    out = {}
    for (b, h) in heads:
        out[(b, h)] = attention(q[b, h], k[b, h], v[b, h], scale, causal, rows, threads, lib)
    return out


def online_blocks(s, v, blocks: Sequence[tuple[int, int]], lib=None):
    """s [n] scores, v [n,dv], blocks = [(start, length), ...] in processing order.
    Returns (m, l, o [dv], lse)."""
    lib = lib or load()
    s = _f64(s).reshape(-1)
    v = _f64(v)
    if v.ndim == 1:
        v = v.reshape(-1, 1)
    n, dv = v.shape
    assert s.shape[0] == n
    st = np.ascontiguousarray(np.array([b[0] for b in blocks], dtype=np.int64))
    ln = np.ascontiguousarray(np.array([b[1] for b in blocks], dtype=np.int64))
    m = ctypes.c_double()
    l = ctypes.c_double()
    lse = ctypes.c_double()
    o = np.empty((dv,), dtype=np.float64)
    rc = lib.oracle_online_blocks(_ptr(s), _ptr(v), n, dv, _ptr(st, _ip), _ptr(ln, _ip), len(blocks),
                                  ctypes.byref(m), ctypes.byref(l), _ptr(o), ctypes.byref(lse))
    if rc != 0:
        raise ValueError("oracle_online_blocks: bad argument")
    return m.value, l.value, o, lse.value


def merge(m, l, o, lib=None):
    """Parts: m [P], l [P], o [P,dv] (normalised).  Returns (m, l, o [dv], lse)."""
    lib = lib or load()
    m = _f64(m).reshape(-1)
    l = _f64(l).reshape(-1)
    o = _f64(o)
    if o.ndim == 1:
        o = o.reshape(-1, 1)
    P, dv = o.shape
    assert m.shape[0] == P and l.shape[0] == P
    mo = ctypes.c_double()
    lo = ctypes.c_double()
    lse = ctypes.c_double()
    oo = np.empty((dv,), dtype=np.float64)
    rc = lib.oracle_merge(_ptr(m), _ptr(l), _ptr(o), P, dv, ctypes.byref(mo), ctypes.byref(lo),
                          _ptr(oo), ctypes.byref(lse))
    if rc != 0:
        raise ValueError("oracle_merge: bad argument")
    return mo.value, lo.value, oo, lse.value


def e4m3(x, lib=None):
    """Nearest FP8 E4M3 value (ties to even, saturating at 448), elementwise."""
    lib = lib or load()
    x = np.asarray(x, dtype=np.float64)
    return np.vectorize(lambda t: lib.oracle_e4m3(float(t)), otypes=[np.float64])(x)


def attention_fp8(q8, k8, v8, scale: float, q_descale: float = 1.0, k_descale: float = 1.0,
                  v_descale: float = 1.0, causal: bool = False, block: int = 128,
                  rows: Sequence[int] | None = None, lib=None):
    """One head of the FP8 forward with Max_offset = 8 (E4M3 values in q8, k8,
    v8 as any float array).  Returns (o [len(rows), d], lse [len(rows)])."""
    lib = lib or load()
    q, k, v = _f64(q8), _f64(k8), _f64(v8)
    nq, d = q.shape
    nk = k.shape[0]
    assert k.shape == (nk, d) and v.shape == (nk, d)
    if rows is None:
        rows_arr, nrows = None, nq
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = rows_arr.shape[0]
    o = np.empty((nrows, d))
    lse = np.empty(nrows)
    rc = lib.oracle_attention_fp8(_ptr(q), nq, _ptr(k), _ptr(v), nk, d, float(scale), float(q_descale),
                                  float(k_descale), float(v_descale), int(bool(causal)), int(block),
                                  None if rows_arr is None else _ptr(rows_arr, _ip), nrows, _ptr(o),
                                  _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_attention_fp8: bad argument")
    return o, lse


def attention_bwd(q, k, v, dout, scale: float, causal: bool = False, window=None,
                  threads: int | None = None, lib=None):
    """One head: gradients of attention.  q, dout [nq,d]; k, v [nk,d].
    window=(wl, wr) overrides `causal` (causal = (-1, 0)).
    Returns dict(dq, dk, dv, lse, dd) (dd = D_i = <dO_i, O_i>)."""
    lib = lib or load()
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    nq, d = q.shape
    nk = k.shape[0]
    assert k.shape == (nk, d) and v.shape == (nk, d) and dout.shape == (nq, d)
    wl, wr = window if window is not None else ((-1, 0) if causal else (-1, -1))
    dq = np.empty((nq, d))
    dk = np.empty((nk, d))
    dv = np.empty((nk, d))
    lse = np.empty(nq)
    dd = np.empty(nq)
    rc = lib.oracle_attention_bwd(_ptr(q), nq, _ptr(k), _ptr(v), nk, d, float(scale), int(wl), int(wr),
                                  _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(lse), _ptr(dd),
                                  threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_attention_bwd: bad argument")
    return {"dq": dq, "dk": dk, "dv": dv, "lse": lse, "dd": dd}


def softmax_rows(x, rows: Sequence[int] | None = None, threads: int | None = None, lib=None):
    """x [R, C]: softmax_two_pass of every row (or of the listed rows).
    Returns (p [len(rows), C], lse [len(rows)])."""
    lib = lib or load()
    x = np.ascontiguousarray(_f64(x))
    assert x.ndim == 2
    R, C = x.shape
    if rows is None:
        sel, nsel = None, R
    else:
        sel = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nsel = sel.shape[0]
    p = np.empty((nsel, C), dtype=np.float64)
    lse = np.empty(nsel, dtype=np.float64)
    rc = lib.oracle_softmax_rows(_ptr(x), R, C, None if sel is None else _ptr(sel, _ip),
                                 nsel, _ptr(p), _ptr(lse), threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_softmax_rows: bad argument")
    return p, lse


def softmax_two_pass(x, lib=None):
    """Returns (p [n], lse)."""
    lib = lib or load()
    x = _f64(x).reshape(-1)
    p = np.empty_like(x)
    lse = ctypes.c_double()
    rc = lib.oracle_softmax_two_pass(_ptr(x), x.shape[0], _ptr(p), ctypes.byref(lse))
    if rc != 0:
        raise ValueError("oracle_softmax_two_pass: bad argument")
    return p, lse.value
