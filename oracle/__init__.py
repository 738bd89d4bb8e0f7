"""The oracle: plain fp64 CPU attention forward, and a CPU model of the blocked algorithm.

Test infrastructure only. The tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` are the only code that imports this package; the
CUDA library and its Python binding never do, and this package imports nothing
from them. Inputs come from ``fa_inputs`` (random numbers only).

* ``attention`` / ``attention_varlen`` / ``attention_rows*`` wrap the C oracle
  in ``attn_oracle.c`` (fp64 two-pass softmax, see that file for the formula
  and its sources). Inputs are bf16 or fp16 bit patterns (``dtype``); K and V
  may have fewer heads than Q (grouped-query attention: query head h reads
  K/V head h // (H // H_kv)).
* ``lse_combine`` merges partial results over disjoint key sets through their
  LSE (``lse_combine.py``).
* ``attention_backward`` gives the fp64 gradients dQ, dK, dV of the forward for
  an upstream dO (``attn_backward.py``).
* ``online_softmax`` is a separate, slow NumPy model of the blocked update with
  delayed rescaling, used to explain GPU differences and to check that the
  result does not depend on the threshold.

Parity status: every function here is pinned by the ``-m "not gpu"`` tests
against the pages' worked example, closed forms, exact-rational brute force
and float64 SDPA; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_ptr = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into liboracle.so with gcc (host code, any architecture)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-Wall", "-Wextra",
           "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            ci, cd = ctypes.c_int, ctypes.c_double
            lib.oracle_attention_bshd.argtypes = [_ptr, _ptr, _ptr, _i64, _i64, _i64, _i64, _i64,
                                                  _i64, ci, cd, ci, _i64, _ptr, _ptr, ci]
            lib.oracle_attention_varlen.argtypes = [_ptr, _ptr, _ptr, _ptr, _i64, _i64, _i64, _i64,
                                                    ci, cd, ci, _ptr, _ptr, ci]
            lib.oracle_attention_rows_bshd.argtypes = [_ptr, _ptr, _ptr, _i64, _i64, _i64, _i64,
                                                       _i64, _i64, ci, cd, ci, _i64, _ptr, _i64,
                                                       _ptr, _ptr, ci]
            lib.oracle_attention_rows_varlen.argtypes = [_ptr, _ptr, _ptr, _ptr, _i64, _i64, _i64,
                                                         _i64, ci, cd, ci, _ptr, _i64, _ptr, _ptr,
                                                         ci]
            for f in (lib.oracle_attention_bshd, lib.oracle_attention_varlen,
                      lib.oracle_attention_rows_bshd, lib.oracle_attention_rows_varlen):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


_DTYPES = {"bf16": 0, "f16": 1}


def _u16(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are bf16 / fp16 bit patterns (uint16)")
    return a


def _dtype(dtype: str) -> int:
    if dtype not in _DTYPES:
        raise ValueError(f"dtype must be one of {sorted(_DTYPES)}")
    return _DTYPES[dtype]


def _heads(H: int, Hkv: int):
    if Hkv < 1 or H % Hkv:
        raise ValueError("the number of query heads must be a multiple of the K/V heads")


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc):
    if rc == -1:
        raise ValueError("oracle: invalid arguments")
    if rc != 0:
        raise MemoryError("oracle: allocation failed")


def attention(q, k, v, scale: float, causal: bool, off: int | None = None, threads: int | None = None,
              dtype: str = "bf16"):
    """q [B,Nq,H,d], k/v [B,Nkv,H_kv,d] bit patterns -> (o [B,Nq,H,d] f64, lse [B,H,Nq] f64).

    ``off`` is the causal diagonal offset; None means N_kv - N_q (bottom-right aligned)."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    B, Nq, H, d = q.shape
    Nkv, Hkv = k.shape[1], k.shape[2]
    if k.shape != (B, Nkv, Hkv, d) or v.shape != k.shape:
        raise ValueError("shape mismatch")
    _heads(H, Hkv)
    off = Nkv - Nq if off is None else int(off)
    o = np.empty((B, Nq, H, d), dtype=np.float64)
    lse = np.empty((B, H, Nq), dtype=np.float64)
    _check(_load().oracle_attention_bshd(_p(q), _p(k), _p(v), B, H, Hkv, Nq, Nkv, d, _dtype(dtype),
                                         float(scale), int(bool(causal)), off, _p(o), _p(lse),
                                         threads or default_threads()))
    return o, lse


def attention_varlen(q, k, v, cu_seqlens, scale: float, causal: bool, threads: int | None = None,
                     dtype: str = "bf16"):
    """Packed q [T,H,d], k/v [T,H_kv,d] bit patterns, cu_seqlens int32 [S+1] -> (o [T,H,d], lse [H,T])."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    T, H, d = q.shape
    Hkv = k.shape[1]
    if k.shape != (T, Hkv, d) or v.shape != k.shape:
        raise ValueError("shape mismatch")
    _heads(H, Hkv)
    if int(cu[-1]) != T:
        raise ValueError("cu_seqlens[-1] must equal the number of packed rows")
    o = np.empty((T, H, d), dtype=np.float64)
    lse = np.empty((H, T), dtype=np.float64)
    _check(_load().oracle_attention_varlen(_p(q), _p(k), _p(v), _p(cu), len(cu) - 1, H, Hkv, d,
                                           _dtype(dtype), float(scale), int(bool(causal)), _p(o),
                                           _p(lse), threads or default_threads()))
    return o, lse


def attention_rows(q, k, v, rows, scale: float, causal: bool, off: int | None = None,
                   threads: int | None = None, dtype: str = "bf16"):
    """Selected rows of the fixed-length problem. rows: int64 [n,3] of (b, h, i) (h a query head).
    Returns (o [n,d], lse [n])."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    B, Nq, H, d = q.shape
    Nkv, Hkv = k.shape[1], k.shape[2]
    if k.shape != (B, Nkv, Hkv, d) or v.shape != k.shape:
        raise ValueError("shape mismatch")
    _heads(H, Hkv)
    off = Nkv - Nq if off is None else int(off)
    rows = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 3)
    o = np.empty((len(rows), d), dtype=np.float64)
    lse = np.empty(len(rows), dtype=np.float64)
    _check(_load().oracle_attention_rows_bshd(_p(q), _p(k), _p(v), B, H, Hkv, Nq, Nkv, d,
                                              _dtype(dtype), float(scale), int(bool(causal)), off,
                                              _p(rows), len(rows), _p(o), _p(lse),
                                              threads or default_threads()))
    return o, lse


def attention_rows_varlen(q, k, v, cu_seqlens, rows, scale: float, causal: bool,
                          threads: int | None = None, dtype: str = "bf16"):
    """Selected rows of the packed problem. rows: int64 [n,2] of (h, token) (h a query head)."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    T, H, d = q.shape
    Hkv = k.shape[1]
    if k.shape != (T, Hkv, d) or v.shape != k.shape:
        raise ValueError("shape mismatch")
    _heads(H, Hkv)
    rows = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 2)
    o = np.empty((len(rows), d), dtype=np.float64)
    lse = np.empty(len(rows), dtype=np.float64)
    _check(_load().oracle_attention_rows_varlen(_p(q), _p(k), _p(v), _p(cu), len(cu) - 1, H, Hkv,
                                                d, _dtype(dtype), float(scale), int(bool(causal)),
                                                _p(rows), len(rows), _p(o), _p(lse),
                                                threads or default_threads()))
    return o, lse


from .attn_backward import attention_backward, attention_backward_varlen, attention_forward  # noqa: E402,F401
from .lse_combine import lse_combine  # noqa: E402,F401
from .online_softmax import online_softmax_rows  # noqa: E402,F401
