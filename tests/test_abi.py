"""The C ABI without a GPU: the library builds, loads, exports every declared
symbol, and rejects bad arguments before touching a device."""
import ctypes
import math
import os
import re

import pytest

import attention_forward_tma_gb300 as fa
from attention_forward_tma_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in ("fa.h", "fa_selftest.h"):
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(fa_\w+)\s*\(", text, flags=re.M))
    return names


def test_headers_declare_the_boundary():
    names = declared_functions()
    assert {"fa_fwd", "fa_fwd_varlen", "fa_error_string", "fa_last_device_status"} <= names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(_build.build())
    for name in sorted(declared_functions()):
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_binding_signatures_cover_the_headers():
    assert declared_functions() == set(fa._SIGNATURES)


def test_error_strings_and_version():
    lib = fa.library()
    for code in range(6):
        assert fa.error_string(code)
    assert fa.error_string(99) == "unknown status"
    assert lib.fa_version() >= 100


def test_release_cached_memory_without_a_pool():
    """No call has allocated from the library's pool in this process: nothing to release,
    and no CUDA call is made."""
    assert fa.library().fa_release_cached_memory() == fa.FA_OK
    fa.release_cached_memory()


NULL = None


def fwd(**kw):
    args = dict(q=16, k=16, v=16, o=16, lse=NULL, B=1, H=1, N=128, d=128, scale=0.125, causal=0, stream=NULL)
    args.update(kw)
    return fa.library().fa_fwd(args["q"], args["k"], args["v"], args["o"], args["lse"], args["B"], args["H"],
                               args["N"], args["d"], args["scale"], args["causal"], args["stream"])


@pytest.mark.parametrize("kw", [dict(q=NULL), dict(k=NULL), dict(v=NULL), dict(o=NULL), dict(q=8),
                                dict(o=24), dict(lse=2), dict(B=0), dict(H=-1), dict(N=0),
                                dict(scale=0.0), dict(scale=-1.0), dict(scale=math.inf), dict(scale=math.nan),
                                dict(causal=2), dict(B=1 << 16, N=1 << 16)])
def test_fwd_rejects_invalid_arguments(kw):
    assert fwd(**kw) == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("d", [0, 32, 96, 256])
def test_fwd_rejects_unsupported_head_dim(d):
    assert fwd(d=d) == fa.FA_ERR_UNSUPPORTED


def varlen(**kw):
    args = dict(q=16, k=16, v=16, o=16, lse=NULL, cu=16, S=2, T=256, maxL=200, H=2, d=64, scale=0.125,
                causal=1, stream=NULL)
    args.update(kw)
    return fa.library().fa_fwd_varlen(args["q"], args["k"], args["v"], args["o"], args["lse"], args["cu"],
                                      args["S"], args["T"], args["maxL"], args["H"], args["d"], args["scale"],
                                      args["causal"], args["stream"])


@pytest.mark.parametrize("kw", [dict(cu=NULL), dict(cu=2), dict(q=NULL), dict(S=0), dict(T=0), dict(maxL=0),
                                dict(H=0), dict(scale=0.0), dict(causal=-1), dict(T=1 << 30, H=8)])
def test_varlen_rejects_invalid_arguments(kw):
    assert varlen(**kw) == fa.FA_ERR_INVALID_ARG


def test_varlen_rejects_unsupported_head_dim():
    assert varlen(d=80) == fa.FA_ERR_UNSUPPORTED


def gqa(**kw):
    args = dict(q=16, k=16, v=16, o=16, lse=NULL, B=1, H=8, Hkv=2, N=128, d=128, scale=0.125, causal=0, dtype=0,
                stream=NULL)
    args.update(kw)
    return fa.library().fa_fwd_gqa(args["q"], args["k"], args["v"], args["o"], args["lse"], args["B"], args["H"],
                                   args["Hkv"], args["N"], args["d"], args["scale"], args["causal"], args["dtype"],
                                   args["stream"])


def varlen_gqa(**kw):
    args = dict(q=16, k=16, v=16, o=16, lse=NULL, cu=16, S=2, T=256, maxL=200, H=8, Hkv=2, d=64, scale=0.125,
                causal=1, dtype=1, stream=NULL)
    args.update(kw)
    return fa.library().fa_fwd_varlen_gqa(args["q"], args["k"], args["v"], args["o"], args["lse"], args["cu"],
                                          args["S"], args["T"], args["maxL"], args["H"], args["Hkv"], args["d"],
                                          args["scale"], args["causal"], args["dtype"], args["stream"])


@pytest.mark.parametrize("kw", [dict(Hkv=0), dict(Hkv=-2), dict(H=8, Hkv=3), dict(H=2, Hkv=4), dict(dtype=2),
                                dict(dtype=-1), dict(q=NULL), dict(k=8), dict(B=0), dict(N=0), dict(scale=0.0),
                                dict(causal=3)])
def test_gqa_rejects_invalid_arguments(kw):
    assert gqa(**kw) == fa.FA_ERR_INVALID_ARG
    if not set(kw) & {"B", "N"}:   # the varlen call has no B, N
        assert varlen_gqa(**kw) == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("H,Hkv", [(6, 2), (12, 1), (256, 1), (144, 3)])
def test_gqa_rejects_group_sizes_that_do_not_divide_the_tile(H, Hkv):
    # G = H / H_kv must be a power of two up to 128
    assert gqa(H=H, Hkv=Hkv) == fa.FA_ERR_UNSUPPORTED
    assert varlen_gqa(H=H, Hkv=Hkv) == fa.FA_ERR_UNSUPPORTED


def test_gqa_rejects_unsupported_head_dim():
    assert gqa(d=96) == fa.FA_ERR_UNSUPPORTED
    assert varlen_gqa(d=256) == fa.FA_ERR_UNSUPPORTED


def fwd_kv(**kw):
    args = dict(q=16, k=16, v=16, o=16, lse=NULL, B=1, H=8, Hkv=2, Nq=1, Nk=4096, d=128, scale=0.125, causal=1,
                dtype=0, splits=0, stream=NULL)
    args.update(kw)
    return fa.library().fa_fwd_kv(*[args[n] for n in ("q", "k", "v", "o", "lse", "B", "H", "Hkv", "Nq", "Nk", "d",
                                                      "scale", "causal", "dtype", "splits", "stream")])


def varlen_kv(**kw):
    args = dict(q=16, k=16, v=16, o=16, lse=NULL, cuq=16, cuk=32, S=2, Tq=2, Tk=9000, maxq=1, maxk=5000, H=8,
                Hkv=2, d=128, scale=0.125, causal=1, dtype=0, splits=4, stream=NULL)
    args.update(kw)
    return fa.library().fa_fwd_varlen_kv(*[args[n] for n in ("q", "k", "v", "o", "lse", "cuq", "cuk", "S", "Tq",
                                                             "Tk", "maxq", "maxk", "H", "Hkv", "d", "scale",
                                                             "causal", "dtype", "splits", "stream")])


def kv_partial(**kw):
    args = dict(q=16, k=16, v=16, o=16, l=16, B=1, H=8, Hkv=2, Nq=100, Nk=1000, Nt=4000, off=1000, d=128,
                scale=0.125, causal=1, dtype=0, stream=NULL)
    args.update(kw)
    return fa.library().fa_fwd_kv_partial(*[args[n] for n in ("q", "k", "v", "o", "l", "B", "H", "Hkv", "Nq", "Nk",
                                                              "Nt", "off", "d", "scale", "causal", "dtype",
                                                              "stream")])


@pytest.mark.parametrize("kw", [dict(off=-1), dict(off=3001), dict(Nt=999), dict(Nk=0), dict(o=NULL), dict(l=NULL),
                                dict(o=8), dict(l=2), dict(Nq=0), dict(Hkv=3), dict(causal=2), dict(dtype=4),
                                dict(scale=0.0), dict(k=NULL)])
def test_kv_partial_rejects_invalid_arguments(kw):
    assert kv_partial(**kw) == fa.FA_ERR_INVALID_ARG


def test_kv_partial_head_dim_and_no_device():
    assert kv_partial(d=96) == fa.FA_ERR_UNSUPPORTED
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        assert kv_partial() == fa.FA_ERR_NO_DEVICE
        assert kv_partial(off=3000) == fa.FA_ERR_NO_DEVICE       # the last shard: ends at the last key
        assert kv_partial(causal=0, off=0, Nt=1000) == fa.FA_ERR_NO_DEVICE


def combine(**kw):
    args = dict(o=16, l=16, P=3, B=1, N=10, H=4, d=128, out=16, lse=NULL, dtype=0, stream=NULL)
    args.update(kw)
    return fa.library().fa_lse_combine(*[args[n] for n in ("o", "l", "P", "B", "N", "H", "d", "out", "lse", "dtype",
                                                           "stream")])


@pytest.mark.parametrize("kw", [dict(Nq=0), dict(Nk=0), dict(splits=-1), dict(Hkv=3), dict(k=NULL), dict(o=8),
                                dict(dtype=5), dict(causal=2), dict(B=1 << 16, Nk=1 << 16)])
def test_fwd_kv_rejects_invalid_arguments(kw):
    assert fwd_kv(**kw) == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [dict(cuk=NULL), dict(cuk=2), dict(Tk=0), dict(maxq=0), dict(maxk=-1),
                                dict(splits=-2), dict(Hkv=16), dict(dtype=3)])
def test_varlen_kv_rejects_invalid_arguments(kw):
    assert varlen_kv(**kw) == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [dict(o=NULL), dict(l=NULL), dict(out=NULL), dict(o=4), dict(out=8), dict(P=0),
                                dict(B=0), dict(N=0), dict(H=0), dict(dtype=2), dict(N=1 << 20, H=1 << 12)])
def test_lse_combine_rejects_invalid_arguments(kw):
    assert combine(**kw) == fa.FA_ERR_INVALID_ARG


def bwd(**kw):
    args = dict(q=16, k=16, v=16, o=16, do=16, lse=16, dq=16, dk=16, dv=16, B=2, H=8, Hkv=2, Nq=300, Nk=200,
                d=128, scale=0.125, causal=1, dtype=0, stream=NULL)
    args.update(kw)
    return fa.library().fa_bwd(*[args[n] for n in ("q", "k", "v", "o", "do", "lse", "dq", "dk", "dv", "B", "H",
                                                   "Hkv", "Nq", "Nk", "d", "scale", "causal", "dtype", "stream")])


def bwd_varlen(**kw):
    args = dict(q=16, k=16, v=16, o=16, do=16, lse=16, dq=16, dk=16, dv=16, cuq=16, cuk=32, S=3, Tq=700,
                Tk=900, maxq=400, maxk=500, H=8, Hkv=2, d=128, scale=0.125, causal=1, dtype=0, stream=NULL)
    args.update(kw)
    return fa.library().fa_bwd_varlen(*[args[n] for n in ("q", "k", "v", "o", "do", "lse", "dq", "dk", "dv", "cuq",
                                                          "cuk", "S", "Tq", "Tk", "maxq", "maxk", "H", "Hkv", "d",
                                                          "scale", "causal", "dtype", "stream")])


@pytest.mark.parametrize("kw", [dict(q=NULL), dict(do=NULL), dict(lse=NULL), dict(dq=NULL), dict(dk=NULL),
                                dict(dv=NULL), dict(o=8), dict(dq=24), dict(lse=2), dict(B=0), dict(Nq=0),
                                dict(Nk=-1), dict(H=6, Hkv=4), dict(scale=0.0), dict(scale=math.nan),
                                dict(causal=3), dict(dtype=2), dict(B=1 << 16, Nq=1 << 16)])
def test_bwd_rejects_invalid_arguments(kw):
    assert bwd(**kw) == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [dict(cuq=NULL), dict(cuk=NULL), dict(cuk=2), dict(dv=NULL), dict(S=0),
                                dict(Tq=0), dict(Tk=0), dict(maxq=0), dict(maxk=0), dict(H=6, Hkv=4),
                                dict(dtype=7), dict(causal=-1), dict(scale=-2.0)])
def test_bwd_varlen_rejects_invalid_arguments(kw):
    assert bwd_varlen(**kw) == fa.FA_ERR_INVALID_ARG


def test_split_queries_reject_invalid_arguments():
    lib = fa.library()
    n = ctypes.c_int(0)
    assert lib.fa_fwd_kv_splits(1, 8, 2, 100, 100, 128, 2, 0, ctypes.byref(n)) == fa.FA_ERR_INVALID_ARG  # causal 2
    assert lib.fa_fwd_kv_splits(1, 8, 2, 100, 100, 128, 1, -1, ctypes.byref(n)) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_fwd_kv_splits(1, 8, 2, 0, 100, 128, 1, 0, ctypes.byref(n)) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_fwd_kv_splits(1, 8, 2, 100, 100, 128, 1, 0, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_fwd_kv_splits(1, 8, 2, 100, 100, 96, 1, 0, ctypes.byref(n)) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_fwd_varlen_kv_splits(0, 10, 100, 8, 2, 0, ctypes.byref(n)) == fa.FA_ERR_INVALID_ARG


def test_new_entry_points_reject_unsupported_head_dim():
    assert bwd(d=96) == fa.FA_ERR_UNSUPPORTED
    assert bwd_varlen(d=256) == fa.FA_ERR_UNSUPPORTED
    assert bwd(H=144, Hkv=3) == fa.FA_ERR_UNSUPPORTED        # a group of 48 rows does not divide the tile
    assert bwd_varlen(H=144, Hkv=3) == fa.FA_ERR_UNSUPPORTED
    assert fwd_kv(d=32) == fa.FA_ERR_UNSUPPORTED
    assert varlen_kv(d=96) == fa.FA_ERR_UNSUPPORTED
    assert combine(d=256) == fa.FA_ERR_UNSUPPORTED


def test_valid_arguments_without_gpu_report_no_device():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert fwd() == fa.FA_ERR_NO_DEVICE
    assert varlen() == fa.FA_ERR_NO_DEVICE
    for H, Hkv in ((8, 2), (128, 1), (4, 4)):
        for dtype in (0, 1):
            assert gqa(H=H, Hkv=Hkv, dtype=dtype) == fa.FA_ERR_NO_DEVICE
            assert varlen_gqa(H=H, Hkv=Hkv, dtype=dtype) == fa.FA_ERR_NO_DEVICE
    for splits in (0, 1, 3, 1000):
        assert fwd_kv(splits=splits) == fa.FA_ERR_NO_DEVICE
        assert varlen_kv(splits=splits) == fa.FA_ERR_NO_DEVICE
    assert fwd_kv(Nq=300, Nk=100) == fa.FA_ERR_NO_DEVICE       # rows without keys are allowed
    assert combine() == fa.FA_ERR_NO_DEVICE
    for dtype in (0, 1):
        assert bwd(dtype=dtype) == fa.FA_ERR_NO_DEVICE
        assert bwd_varlen(dtype=dtype) == fa.FA_ERR_NO_DEVICE
    assert bwd(H=4, Hkv=4, d=64, causal=0) == fa.FA_ERR_NO_DEVICE


@pytest.mark.parametrize("opt,val,ok", [(1, 8.0, True), (1, 0.0, True), (1, 1e30, True), (1, -1.0, False),
                                        (1, math.nan, False), (2, 1e9, True), (2, 10.0, False),
                                        (3, 1, True), (3, 0, True), (3, -1, True), (3, 2, True), (3, 3, False),
                                        (4, 0, True), (4, 8, True), (4, 9, False), (4, 2.5, False),
                                        (5, 0, True), (5, 1, True), (5, 2, False), (5, 0.5, False),
                                        (6, 0, True), (6, 1, True), (6, -1, False),
                                        (7, 0, True), (7, 1, True), (7, 3, False),
                                        (8, 0, True), (8, 12, True), (8, -1, False), (8, 1.5, False),
                                        (9, -1, True), (9, 0, True), (9, 1, True), (9, 2, False), (9, 0.5, False),
                                        (99, 1, False)])
def test_set_option_validation(opt, val, ok):
    lib = fa.library()
    st = lib.fa_set_option(opt, val)
    assert (st == fa.FA_OK) == ok
    # restore defaults
    lib.fa_set_option(1, 8.0)
    lib.fa_set_option(2, 2e9)
    lib.fa_set_option(3, -1)
    lib.fa_set_option(4, 0)
    lib.fa_set_option(5, 0)
    lib.fa_set_option(6, 0)
    lib.fa_set_option(7, 1)
    lib.fa_set_option(8, 0)
    lib.fa_set_option(9, -1)
