"""Attention forward for NVIDIA GB300 (sm_103a): Python binding of libfa_gb300.so.

This module only marshals arguments: it checks dtypes and shapes of torch
tensors, passes their device pointers and the current CUDA stream to the C ABI
declared in ``include/fa.h`` and ``include/fa_selftest.h``, and turns status
codes into exceptions. Every step of the computation runs in the library's CUDA
kernels; there is no CPU path. If the library cannot be built or loaded, or no
sm_103 GPU is present, the calls raise.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

from . import _build

__all__ = ["fa_fwd", "fa_fwd_varlen", "fa_fwd_kv_partial", "fa_bwd", "fa_bwd_varlen", "lse_combine", "num_splits", "num_splits_varlen", "FaError", "set_option", "last_device_status", "library",
           "release_cached_memory",
           "FA_DTYPE_BF16", "FA_DTYPE_FP16",
           "selftest_mma_tile", "selftest_exp2", "selftest_wait_timeout", "varlen_schedule",
           "FA_OK", "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED", "FA_ERR_CUDA", "FA_ERR_TIMEOUT",
           "FA_ERR_NO_DEVICE", "FA_ERR_CAPACITY"]

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT, FA_ERR_NO_DEVICE, FA_ERR_CAPACITY = range(7)
FA_DTYPE_BF16, FA_DTYPE_FP16 = 0, 1
_OPTIONS = {"tau": 1, "wait_timeout_ns": 2, "persistent": 3, "exp2_emulation": 4, "bwd_deterministic": 5,
            "softmax_stagger": 6, "stats_tmem": 7, "bwd_section": 8, "solo_tiles": 9}

_vp, _ci, _cf = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
_SIGNATURES = {
    "fa_fwd": [_vp, _vp, _vp, _vp, _vp, _ci, _ci, _ci, _ci, _cf, _ci, _vp],
    "fa_fwd_gqa": [_vp, _vp, _vp, _vp, _vp, _ci, _ci, _ci, _ci, _ci, _cf, _ci, _ci, _vp],
    "fa_fwd_kv": [_vp, _vp, _vp, _vp, _vp, _ci, _ci, _ci, _ci, _ci, _ci, _cf, _ci, _ci, _ci, _vp],
    "fa_fwd_varlen": [_vp, _vp, _vp, _vp, _vp, _vp, _ci, _ci, _ci, _ci, _ci, _cf, _ci, _vp],
    "fa_fwd_varlen_gqa": [_vp, _vp, _vp, _vp, _vp, _vp, _ci, _ci, _ci, _ci, _ci, _ci, _cf, _ci, _ci, _vp],
    "fa_fwd_varlen_kv": [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _ci, _ci, _ci, _ci, _ci, _ci, _ci, _ci, _cf, _ci, _ci,
                         _ci, _vp],
    "fa_lse_combine": [_vp, _vp, _ci, _ci, _ci, _ci, _ci, _vp, _vp, _ci, _vp],
    "fa_fwd_kv_partial": [_vp, _vp, _vp, _vp, _vp, _ci, _ci, _ci, _ci, _ci, _ci, _ci, _ci, _cf, _ci, _ci, _vp],
    "fa_bwd": [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _ci, _ci, _ci, _ci, _ci, _ci, _cf, _ci, _ci, _vp],
    "fa_bwd_varlen": [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _ci, _ci, _ci, _ci, _ci, _ci, _ci, _ci,
                      _cf, _ci, _ci, _vp],
    "fa_fwd_kv_splits": [_ci, _ci, _ci, _ci, _ci, _ci, _ci, _ci, ctypes.POINTER(_ci)],
    "fa_fwd_varlen_kv_splits": [_ci, _ci, _ci, _ci, _ci, _ci, ctypes.POINTER(_ci)],
    "fa_fwd_varlen_noalloc": [_vp, _vp, _vp, _vp, _vp, _vp, _ci, _ci, _ci, _ci, _ci, _cf, _ci, _vp],
    "fa_error_string": [_ci],
    "fa_last_device_status": [_vp, ctypes.POINTER(ctypes.c_ulonglong)],
    "fa_set_option": [_ci, ctypes.c_double],
    "fa_version": [],
    "fa_release_cached_memory": [],
    "fa_selftest_mma_tile": [_vp, _vp, _vp, _vp, _vp, _vp, _ci, _ci, _vp],
    "fa_selftest_exp2": [_vp, _vp, _ci, _ci, _vp],
    "fa_selftest_wait_timeout": [ctypes.c_ulonglong, _vp],
    "fa_varlen_schedule": [_vp, _vp, _ci, _ci, _ci, _ci, _ci, _ci, _vp, _vp, _vp],
    "fa_trace_configure": [_vp, _ci],
    "fa_trace_layout": [ctypes.POINTER(_ci), ctypes.POINTER(_ci)],
}

_lock = threading.Lock()
_lib = None


class FaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {error_string(status)} (status {status})")


def library() -> ctypes.CDLL:
    """Load (building first if needed) the in-tree libfa_gb300.so, or its tracing
    build libfa_gb300_trace.so when the environment sets FA_GB300_TRACE=1."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            path = _build.build(trace=os.environ.get("FA_GB300_TRACE", "0") == "1")
            lib = ctypes.CDLL(path)
            for name, args in _SIGNATURES.items():
                f = getattr(lib, name)
                f.argtypes = args
                f.restype = ctypes.c_char_p if name == "fa_error_string" else ctypes.c_int
            _lib = lib
    return _lib


def error_string(status: int) -> str:
    return library().fa_error_string(int(status)).decode()


def _check(status: int, what: str):
    if status != FA_OK:
        raise FaError(status, what)


def set_option(name: str, value: float) -> None:
    """Process-wide knobs: tau, wait_timeout_ns, persistent (-1/0/1/2), exp2_emulation (0..8),
    bwd_deterministic, softmax_stagger, stats_tmem (0/1), bwd_section (0 = automatic),
    solo_tiles (-1 = automatic, 0, 1)."""
    _check(library().fa_set_option(_OPTIONS[name], float(value)), f"set_option({name})")


def _torch():
    import torch
    return torch


def _stream_handle(stream, device):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, name, dtype, ndim=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    allowed = dtype if isinstance(dtype, tuple) else (dtype,)
    if t.dtype not in allowed:
        raise TypeError(f"{name} must be {' or '.join(map(str, allowed))}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions")


def _dtype_code(q):
    torch = _torch()
    _need(q, "q", (torch.bfloat16, torch.float16))
    return FA_DTYPE_FP16 if q.dtype == torch.float16 else FA_DTYPE_BF16


def fa_fwd(q, k, v, *, scale: float | None = None, causal: bool = False, out=None, lse=None,
           return_lse: bool = True, num_splits: int = 1, stream=None):
    """Attention forward: q [B, N_q, H, d], k and v [B, N_kv, H_kv, d], all bf16 or all fp16.
    Returns (o, lse) or o; o has q's shape and type.

    H_kv < H is grouped-query attention (query head h uses K/V head h // (H // H_kv));
    H // H_kv must be a power of two up to 128. N_kv may differ from N_q; the causal
    mask is bottom-right aligned (query i sees keys j <= i + N_kv - N_q). lse is fp32
    [B, H, N_q] (natural log of the scaled logits' sum of exponentials). scale
    defaults to 1/sqrt(d). num_splits > 1 cuts the keys into ranges computed in
    parallel and merged through their LSE (0: the library decides)."""
    torch = _torch()
    _need(q, "q", (torch.bfloat16, torch.float16), 4)
    code = FA_DTYPE_FP16 if q.dtype == torch.float16 else FA_DTYPE_BF16
    B, N, H, d = q.shape
    Nk, Hkv = (k.shape[1], k.shape[2]) if isinstance(k, torch.Tensor) and k.dim() == 4 else (N, H)
    for name, t in (("k", k), ("v", v)):
        _need(t, name, q.dtype, 4)
        if tuple(t.shape) != (B, Nk, Hkv, d):
            raise ValueError(f"{name} must have shape {(B, Nk, Hkv, d)}")
    if out is None:
        out = torch.empty_like(q)
    else:
        _need(out, "out", q.dtype, 4)
        if tuple(out.shape) != (B, N, H, d):
            raise ValueError("out has the wrong shape")
    if lse is None and return_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    elif lse is not None:
        _need(lse, "lse", torch.float32, 3)
        if tuple(lse.shape) != (B, H, N):
            raise ValueError("lse must have shape (B, H, N)")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = library().fa_fwd_kv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                             lse.data_ptr() if lse is not None else None, B, H, Hkv, N, Nk, d, scale,
                             int(bool(causal)), code, int(num_splits), _stream_handle(stream, q.device))
    _check(st, "fa_fwd")
    return (out, lse) if lse is not None else out


def fa_fwd_varlen(q, k, v, cu_seqlens, max_seqlen: int, *, scale: float | None = None, causal: bool = False,
                  out=None, lse=None, return_lse: bool = True, cu_seqlens_k=None, max_seqlen_k: int | None = None,
                  num_splits: int = 1, stream=None):
    """Packed variable-length attention forward: q [T, H, d], k and v [T_kv, H_kv, d] (bf16 or fp16);
    cu_seqlens int32 [S+1] on the device (query rows; also the key rows unless
    cu_seqlens_k is given). Returns (o, lse) or o; lse is fp32 [H, T]."""
    torch = _torch()
    code = _dtype_code(q)
    _need(q, "q", q.dtype, 3)
    T, H, d = q.shape
    Tk, Hkv = (k.shape[0], k.shape[1]) if isinstance(k, torch.Tensor) and k.dim() == 3 else (T, H)
    for name, t in (("k", k), ("v", v)):
        _need(t, name, q.dtype, 3)
        if tuple(t.shape) != (Tk, Hkv, d):
            raise ValueError(f"{name} must have shape {(Tk, Hkv, d)}")
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    if cu_seqlens_k is None:
        if Tk != T:
            raise ValueError("k and v must have q's rows unless cu_seqlens_k is given")
        cu_seqlens_k = cu_seqlens
    else:
        _need(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1)
        if cu_seqlens_k.numel() != cu_seqlens.numel():
            raise ValueError("cu_seqlens_k must have as many entries as cu_seqlens")
    max_seqlen_k = int(max_seqlen) if max_seqlen_k is None else int(max_seqlen_k)
    if out is None:
        out = torch.empty_like(q)
    else:
        _need(out, "out", q.dtype, 3)
    if lse is None and return_lse:
        lse = torch.empty((H, T), dtype=torch.float32, device=q.device)
    elif lse is not None:
        _need(lse, "lse", torch.float32, 2)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = library().fa_fwd_varlen_kv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                    lse.data_ptr() if lse is not None else None, cu_seqlens.data_ptr(),
                                    cu_seqlens_k.data_ptr(), cu_seqlens.numel() - 1, T, Tk, int(max_seqlen),
                                    max_seqlen_k, H, Hkv, d, scale, int(bool(causal)), code, int(num_splits),
                                    _stream_handle(stream, q.device))
    _check(st, "fa_fwd_varlen")
    return (out, lse) if lse is not None else out


def fa_bwd(q, k, v, o, dout, lse, *, scale: float | None = None, causal: bool = False, dq=None, dk=None, dv=None,
           stream=None):
    """Backward of fa_fwd: q, o, dout [B, N_q, H, d]; k, v [B, N_kv, H_kv, d] (bf16 or fp16);
    lse fp32 [B, H, N_q] as returned by fa_fwd for the same inputs. Returns (dq, dk, dv)."""
    torch = _torch()
    code = _dtype_code(q)
    _need(q, "q", q.dtype, 4)
    B, N, H, d = q.shape
    if not (isinstance(k, torch.Tensor) and k.dim() == 4):
        raise TypeError("k must be a 4-dimensional torch.Tensor")
    Nk, Hkv = k.shape[1], k.shape[2]
    for name, t, shape in (("k", k, (B, Nk, Hkv, d)), ("v", v, (B, Nk, Hkv, d)), ("o", o, (B, N, H, d)),
                           ("dout", dout, (B, N, H, d))):
        _need(t, name, q.dtype, 4)
        if tuple(t.shape) != shape:
            raise ValueError(f"{name} must have shape {shape}")
    _need(lse, "lse", torch.float32, 3)
    if tuple(lse.shape) != (B, H, N):
        raise ValueError("lse must have shape (B, H, N_q)")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t, ref in (("dq", dq, q), ("dk", dk, k), ("dv", dv, v)):
        _need(t, name, q.dtype, 4)
        if t.shape != ref.shape:
            raise ValueError(f"{name} has the wrong shape")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    _check(library().fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(), lse.data_ptr(),
                            dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Hkv, N, Nk, d, scale,
                            int(bool(causal)), code, _stream_handle(stream, q.device)), "fa_bwd")
    return dq, dk, dv


def fa_bwd_varlen(q, k, v, o, dout, lse, cu_seqlens, max_seqlen: int, *, cu_seqlens_k=None,
                  max_seqlen_k: int | None = None, scale: float | None = None, causal: bool = False, dq=None,
                  dk=None, dv=None, stream=None):
    """Backward of fa_fwd_varlen: q, o, dout [T, H, d]; k, v [T_kv, H_kv, d] (bf16 or fp16);
    lse fp32 [H, T] as returned by fa_fwd_varlen for the same inputs; cu_seqlens (and
    cu_seqlens_k, default cu_seqlens) int32 [S+1] on the device. Returns (dq, dk, dv)."""
    torch = _torch()
    code = _dtype_code(q)
    _need(q, "q", q.dtype, 3)
    T, H, d = q.shape
    if not (isinstance(k, torch.Tensor) and k.dim() == 3):
        raise TypeError("k must be a 3-dimensional torch.Tensor")
    Tk, Hkv = k.shape[0], k.shape[1]
    for name, t, shape in (("k", k, (Tk, Hkv, d)), ("v", v, (Tk, Hkv, d)), ("o", o, (T, H, d)),
                           ("dout", dout, (T, H, d))):
        _need(t, name, q.dtype, 3)
        if tuple(t.shape) != shape:
            raise ValueError(f"{name} must have shape {shape}")
    _need(lse, "lse", torch.float32, 2)
    if tuple(lse.shape) != (H, T):
        raise ValueError("lse must have shape (H, T)")
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    if cu_seqlens_k is None:
        if Tk != T:
            raise ValueError("k and v must have q's rows unless cu_seqlens_k is given")
        cu_seqlens_k = cu_seqlens
    else:
        _need(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1)
        if cu_seqlens_k.numel() != cu_seqlens.numel():
            raise ValueError("cu_seqlens_k must have as many entries as cu_seqlens")
    max_seqlen_k = int(max_seqlen) if max_seqlen_k is None else int(max_seqlen_k)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t, ref in (("dq", dq, q), ("dk", dk, k), ("dv", dv, v)):
        _need(t, name, q.dtype, 3)
        if t.shape != ref.shape:
            raise ValueError(f"{name} has the wrong shape")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    _check(library().fa_bwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
                                   lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), cu_seqlens.data_ptr(),
                                   cu_seqlens_k.data_ptr(), cu_seqlens.numel() - 1, T, Tk, int(max_seqlen),
                                   max_seqlen_k, H, Hkv, d, scale, int(bool(causal)), code,
                                   _stream_handle(stream, q.device)), "fa_bwd_varlen")
    return dq, dk, dv


def fa_fwd_kv_partial(q, k, v, kv_offset: int, n_kv_total: int, *, scale: float | None = None,
                      causal: bool = False, o_part=None, lse_part=None, stream=None):
    """One key shard of a longer sequence: q [B, N_q, H, d]; k, v [B, N_kv, H_kv, d] hold keys
    [kv_offset, kv_offset + N_kv) of a sequence of n_kv_total keys (bf16 or fp16; a causal
    mask is the full sequence's bottom-right one). Returns (o_part fp32 [B, N_q, H, d],
    lse_part fp32 [B, H, N_q]): the output normalised over this shard's keys and its LSE
    (0 and -inf for rows that see none of them), to be merged with lse_combine."""
    torch = _torch()
    code = _dtype_code(q)
    _need(q, "q", q.dtype, 4)
    B, Nq, H, d = q.shape
    for name, t in (("k", k), ("v", v)):
        _need(t, name, q.dtype, 4)
    Nk, Hkv = k.shape[1], k.shape[2]
    if tuple(k.shape) != (B, Nk, Hkv, d) or tuple(v.shape) != tuple(k.shape):
        raise ValueError(f"k and v must have shape {(B, Nk, Hkv, d)}")
    if o_part is None:
        o_part = torch.empty((B, Nq, H, d), dtype=torch.float32, device=q.device)
    if lse_part is None:
        lse_part = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    _need(o_part, "o_part", torch.float32, 4)
    _need(lse_part, "lse_part", torch.float32, 3)
    if tuple(o_part.shape) != (B, Nq, H, d) or tuple(lse_part.shape) != (B, H, Nq):
        raise ValueError("o_part / lse_part have the wrong shape")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    _check(library().fa_fwd_kv_partial(q.data_ptr(), k.data_ptr(), v.data_ptr(), o_part.data_ptr(),
                                       lse_part.data_ptr(), B, H, Hkv, Nq, Nk, int(n_kv_total), int(kv_offset), d,
                                       scale, int(bool(causal)), code, _stream_handle(stream, q.device)),
           "fa_fwd_kv_partial")
    return o_part, lse_part


def lse_combine(o_parts, lse_parts, *, out=None, lse=None, return_lse: bool = True, dtype=None, stream=None):
    """Merge results over disjoint key sets: o_parts fp32 [P, B, N, H, d], lse_parts fp32 [P, B, H, N]
    (-inf: the part saw no key). Returns (o [B, N, H, d] in bf16 (default) or fp16, lse fp32 [B, H, N])."""
    torch = _torch()
    _need(o_parts, "o_parts", torch.float32, 5)
    _need(lse_parts, "lse_parts", torch.float32, 4)
    P, B, N, H, d = o_parts.shape
    if tuple(lse_parts.shape) != (P, B, H, N):
        raise ValueError(f"lse_parts must have shape {(P, B, H, N)}")
    if out is None:
        out = torch.empty((B, N, H, d), dtype=dtype or torch.bfloat16, device=o_parts.device)
    _need(out, "out", (torch.bfloat16, torch.float16), 4)
    if tuple(out.shape) != (B, N, H, d):
        raise ValueError("out has the wrong shape")
    if lse is None and return_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=o_parts.device)
    elif lse is not None:
        _need(lse, "lse", torch.float32, 3)
    code = FA_DTYPE_FP16 if out.dtype == torch.float16 else FA_DTYPE_BF16
    _check(library().fa_lse_combine(o_parts.data_ptr(), lse_parts.data_ptr(), P, B, N, H, d, out.data_ptr(),
                                    lse.data_ptr() if lse is not None else None, code,
                                    _stream_handle(stream, o_parts.device)), "fa_lse_combine")
    return (out, lse) if lse is not None else out


def num_splits(B: int, H: int, H_kv: int, N_q: int, N_kv: int, requested: int = 0, causal: bool = False,
               d: int = 128) -> int:
    """Key ranges fa_fwd would use for these sizes, head dimension and mask with num_splits=requested
    (0: the library's choice)."""
    n = ctypes.c_int(0)
    _check(library().fa_fwd_kv_splits(B, H, H_kv, N_q, N_kv, d, int(bool(causal)), requested, ctypes.byref(n)),
           "fa_fwd_kv_splits")
    return n.value


def num_splits_varlen(num_seqs: int, total_q: int, max_seqlen_k: int, H: int, H_kv: int, requested: int = 0) -> int:
    """Key ranges fa_fwd_varlen would use with num_splits=requested."""
    n = ctypes.c_int(0)
    _check(library().fa_fwd_varlen_kv_splits(num_seqs, total_q, max_seqlen_k, H, H_kv, requested, ctypes.byref(n)),
           "fa_fwd_varlen_kv_splits")
    return n.value


def last_device_status(stream=None):
    """Synchronize the stream; return (status, raw word) of the device-side status, and clear it."""
    torch = _torch()
    word = ctypes.c_ulonglong(0)
    st = library().fa_last_device_status(_stream_handle(stream, torch.device("cuda")), ctypes.byref(word))
    return st, word.value


def release_cached_memory() -> None:
    """Return the library's cached temporary memory (split partials, varlen tile lists,
    backward workspaces) to the system; call after synchronising the streams it ran on."""
    _check(library().fa_release_cached_memory(), "release_cached_memory")


def selftest_mma_tile(q, k, v, p, stream=None):
    """One tile through the MMA plumbing: returns (S = Q K^T fp32 [128,128], O = P V fp32 [128,d]).
    q, k, v, p: all bf16 or all fp16."""
    torch = _torch()
    code = _dtype_code(q)
    for name, t in (("q", q), ("k", k), ("v", v), ("p", p)):
        _need(t, name, q.dtype, 2)
    d = q.shape[1]
    s = torch.empty((128, 128), dtype=torch.float32, device=q.device)
    o = torch.empty((128, d), dtype=torch.float32, device=q.device)
    _check(library().fa_selftest_mma_tile(q.data_ptr(), k.data_ptr(), v.data_ptr(), p.data_ptr(), s.data_ptr(),
                                          o.data_ptr(), d, code, _stream_handle(stream, q.device)),
           "fa_selftest_mma_tile")
    return s, o


def selftest_exp2(x, use_poly: int, stream=None):
    """2^x on the device: use_poly 0 = hardware ex2, 1 = FMA polynomial, 2 = its packed-pair form."""
    torch = _torch()
    _need(x, "x", torch.float32)
    y = torch.empty_like(x)
    _check(library().fa_selftest_exp2(x.data_ptr(), y.data_ptr(), x.numel(), int(use_poly),
                                      _stream_handle(stream, x.device)), "fa_selftest_exp2")
    return y


def selftest_wait_timeout(timeout_ns: int, stream=None) -> int:
    """Returns the status the never-completing wait recorded (FA_ERR_TIMEOUT when correct)."""
    torch = _torch()
    return library().fa_selftest_wait_timeout(int(timeout_ns), _stream_handle(stream, torch.device("cuda")))


def varlen_schedule(cu_seqlens, H: int, causal: bool, capacity: int, stream=None, group: int = 1,
                    cu_seqlens_k=None, splits: int = 1):
    """The longest-first varlen tile list: (tasks int32 [count, 4] of (seq, kv head | range << 16,
    m_block, cost), count). H is the number of K/V heads; group the query heads per K/V head."""
    torch = _torch()
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    cu_seqlens_k = cu_seqlens if cu_seqlens_k is None else cu_seqlens_k
    tasks = torch.full((max(capacity, 1), 4), -1, dtype=torch.int32, device=cu_seqlens.device)
    count = torch.zeros(1, dtype=torch.int32, device=cu_seqlens.device)
    _check(library().fa_varlen_schedule(cu_seqlens.data_ptr(), cu_seqlens_k.data_ptr(), cu_seqlens.numel() - 1, H,
                                        int(group), int(bool(causal)), int(splits),
                                        capacity, tasks.data_ptr(), count.data_ptr(),
                                        _stream_handle(stream, cu_seqlens.device)), "fa_varlen_schedule")
    n = int(count.item())
    return tasks[:n], n
