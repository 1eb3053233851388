"""CPU oracle for scaled dot-product attention (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg use this
package.  It wraps ``oracle.c`` (plain fp64 loops; see that file's header for
the definition it follows and the readings it takes) through ctypes.  It shares
no code with the CUDA library and never imports it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

MASK_NONE, MASK_CAUSAL, MASK_PADDING = 0, 1, 2


def compile_source(src: str, out: str) -> str:
    """Compile a C source of the oracle into a shared library with gcc (C11, -O2)."""
    tmp = out + ".tmp%d" % os.getpid()
    subprocess.check_call(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-pthread",
                           src, "-o", tmp, "-lm"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (skipped when up to date)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        compile_source(_SRC, _LIB_PATH)
    return _LIB_PATH


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        P = ctypes.c_void_p
        I = ctypes.c_int
        I64 = ctypes.c_int64
        D = ctypes.c_double
        lib.oracle_sdpa.argtypes = [P, P, P, P, I, I, I, I, I, I, I, P, D, P, I64, I]
        lib.oracle_sdpa.restype = I
        lib.oracle_mha.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, P, D, P, I64, I]
        lib.oracle_mha.restype = I
        lib.oracle_sdpa_restricted.argtypes = [P, P, P, P, I, I, I, I, I, I, I, P, I, D, P, I64, I]
        lib.oracle_sdpa_restricted.restype = I
        lib.oracle_sdpa_decode.argtypes = [P, P, P, P, I, I, I, I, I, I, P, D, P, I64, I]
        lib.oracle_sdpa_decode.restype = I
        lib.oracle_sdpa_backward.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, D, I, I]
        lib.oracle_sdpa_backward.restype = I
        lib.oracle_sdpa_lse.argtypes = [P, P, P, I, I, I, I, I, I, P, I, D, I]
        lib.oracle_sdpa_lse.restype = I
        self.lib = lib
        self.path = lib_path

    def sdpa(self, *args, **kwargs):
        return _sdpa(self.lib, *args, **kwargs)

    def mha(self, *args, **kwargs):
        return _mha(self.lib, *args, **kwargs)

    def decode(self, *args, **kwargs):
        return _decode(self.lib, *args, **kwargs)

    def backward(self, *args, **kwargs):
        return _backward(self.lib, *args, **kwargs)

    def lse(self, *args, **kwargs):
        return _lse(self.lib, *args, **kwargs)


_default: Oracle | None = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def sdpa(*args, **kwargs):
    """Eq. (1) with masks; see ``_sdpa``.  Uses the library built from oracle.c."""
    return default().sdpa(*args, **kwargs)


def mha(*args, **kwargs):
    """Multi-head attention; see ``_mha``.  Uses the library built from oracle.c."""
    return default().mha(*args, **kwargs)


def backward(*args, **kwargs):
    """Gradients of Eq. (1); see ``_backward``."""
    return default().backward(*args, **kwargs)


def lse(*args, **kwargs):
    """Per-row log of the softmax denominator; see ``_lse``."""
    return default().lse(*args, **kwargs)


def _lse(lib, q, k, mask_kind=MASK_NONE, kv_lengths=None, scale=0.0, window=None, threads=None):
    """lse [b,h,n_q] float64: ln sum over visible keys of exp(scale q.k), -inf
    for a row that sees no key (window=None: plain attention)."""
    q, k = _f32(q), _f32(k)
    b, h, n_q, d_k = q.shape
    n_k = k.shape[2]
    lens = None if kv_lengths is None else np.ascontiguousarray(kv_lengths, dtype=np.int32)
    out = np.zeros((b, h, n_q), dtype=np.float64)
    rc = lib.oracle_sdpa_lse(_ptr(q), _ptr(k), _ptr(out), b, h, n_q, n_k, d_k, int(mask_kind),
                             _ptr(lens), int(window or 0), float(scale),
                             threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_sdpa_lse: bad arguments")
    return out


def _backward(lib, q, k, v, dout, mask_kind=MASK_NONE, kv_lengths=None, scale=0.0, window=None,
              threads=None, out=None):
    """dq, dk, dv (float64, shapes of q, k, v) of sum(dout * attention(q, k, v)).

    ``out`` [b,h,n_q,d_v] is the forward output handed to the backward (None:
    the exact output).  It enters only through D_i = dO_i . O_i in
    dS = P o (dP - D), as it does for a backward routine that takes O as an input.
    """
    q, k, v, dout = _f32(q), _f32(k), _f32(v), _f32(dout)
    b, h, n_q, d_k = q.shape
    n_k, d_v = k.shape[2], v.shape[3]
    if out is not None:
        out = _f32(out)
        assert out.shape == (b, h, n_q, d_v)
    lens = None if kv_lengths is None else np.ascontiguousarray(kv_lengths, dtype=np.int32)
    dq = np.zeros(q.shape, dtype=np.float64)
    dk = np.zeros(k.shape, dtype=np.float64)
    dv = np.zeros(v.shape, dtype=np.float64)
    rc = lib.oracle_sdpa_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(out), _ptr(dq), _ptr(dk),
                                  _ptr(dv), b, h, n_q, n_k, d_k, d_v, int(mask_kind), _ptr(lens),
                                  float(scale), int(window or 0), threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_sdpa_backward rejected its arguments")
    return dq, dk, dv


def decode(*args, **kwargs):
    """One decoding step over a cache; see ``_decode``."""
    return default().decode(*args, **kwargs)


def _decode(lib, q, k, v, kv_lengths=None, scale=0.0, rows=None, threads=None):
    """n_q new queries q [b,h,n_q,d_k] against caches k [b,h,n_k,d_k], v [b,h,n_k,d_v]
    of lengths kv_lengths [b] (None: n_k).  Query i sees keys j <= len_b - n_q + i.
    Returns float64 [b,h,n_q,d_v] (or [len(rows), d_v])."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    b, h, n_q, d_k = q.shape
    n_k, d_v = k.shape[2], v.shape[3]
    lens = None if kv_lengths is None else np.ascontiguousarray(kv_lengths, dtype=np.int32)
    if rows is None:
        out = np.zeros((b, h, n_q, d_v), dtype=np.float64)
        rows_arr, n_rows = None, 0
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n_rows = rows_arr.size
        out = np.zeros((n_rows, d_v), dtype=np.float64)
    rc = lib.oracle_sdpa_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(out), b, h, n_q, n_k, d_k, d_v,
                                _ptr(lens), float(scale), _ptr(rows_arr), n_rows,
                                threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_sdpa_decode rejected its arguments")
    return out


def _sdpa(lib, q, k, v, mask_kind=MASK_NONE, kv_lengths=None, scale=0.0, rows=None, threads=None,
          window=None):
    """Eq. (1) with masks on BHSD arrays q [b,h,n_q,d_k], k [b,h,n_k,d_k], v [b,h,n_k,d_v].

    Returns float64 [b,h,n_q,d_v], or [len(rows), d_v] when ``rows`` (flat ids
    (bi*h + hi)*n_q + i) is given.  ``scale`` <= 0 selects 1/sqrt(d_k).
    ``window`` = r restricts query i to the r keys i - (r-1)//2 .. i + r//2
    (restricted self-attention, section 4).
    """
    q, k, v = _f32(q), _f32(k), _f32(v)
    b, h, n_q, d_k = q.shape
    n_k, d_v = k.shape[2], v.shape[3]
    assert k.shape == (b, h, n_k, d_k) and v.shape == (b, h, n_k, d_v)
    lens = None if kv_lengths is None else np.ascontiguousarray(kv_lengths, dtype=np.int32)
    if rows is None:
        out = np.zeros((b, h, n_q, d_v), dtype=np.float64)
        rows_arr, n_rows = None, 0
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n_rows = rows_arr.size
        out = np.zeros((n_rows, d_v), dtype=np.float64)
    if window is None:
        rc = lib.oracle_sdpa(_ptr(q), _ptr(k), _ptr(v), _ptr(out), b, h, n_q, n_k, d_k, d_v,
                             int(mask_kind), _ptr(lens), float(scale), _ptr(rows_arr), n_rows,
                             threads or default_threads())
    else:
        rc = lib.oracle_sdpa_restricted(_ptr(q), _ptr(k), _ptr(v), _ptr(out), b, h, n_q, n_k,
                                        d_k, d_v, int(mask_kind), _ptr(lens), int(window),
                                        float(scale), _ptr(rows_arr), n_rows,
                                        threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_sdpa rejected its arguments")
    return out


def _mha(lib, xq, xkv, wq, wk, wv, wo, h, d_k, d_v, mask_kind=MASK_NONE, kv_lengths=None, scale=0.0,
        rows=None, threads=None):
    """MultiHead(X_q, X_kv, X_kv) = Concat(head_1..head_h) W^O (section 3.2.2).

    xq [b,n_q,d_model], xkv [b,n_k,d_model]; wq, wk [d_model,h*d_k]; wv [d_model,h*d_v];
    wo [h*d_v,d_model].  Returns float64 [b,n_q,d_model], or [len(rows), d_model]
    for flat row ids bi*n_q + i.
    """
    xq, xkv, wq, wk, wv, wo = map(_f32, (xq, xkv, wq, wk, wv, wo))
    b, n_q, d_model = xq.shape
    n_k = xkv.shape[1]
    assert wq.shape == (d_model, h * d_k) and wk.shape == (d_model, h * d_k)
    assert wv.shape == (d_model, h * d_v) and wo.shape == (h * d_v, d_model)
    lens = None if kv_lengths is None else np.ascontiguousarray(kv_lengths, dtype=np.int32)
    if rows is None:
        out = np.zeros((b, n_q, d_model), dtype=np.float64)
        rows_arr, n_rows = None, 0
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n_rows = rows_arr.size
        out = np.zeros((n_rows, d_model), dtype=np.float64)
    rc = lib.oracle_mha(_ptr(xq), _ptr(xkv), _ptr(wq), _ptr(wk), _ptr(wv), _ptr(wo), _ptr(out),
                            b, n_q, n_k, d_model, h, d_k, d_v, int(mask_kind), _ptr(lens),
                            float(scale), _ptr(rows_arr), n_rows, threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_mha rejected its arguments")
    return out
