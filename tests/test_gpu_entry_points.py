"""The boundary's two named entry points, called by their exact symbols through ctypes.

fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, stream) and
fa_fwd_varlen(q, k, v, o, lse, cu_seqlens, num_seqs, total_tokens, max_seqlen, H, d,
scale, causal, stream) are the interface the library's header declares for the
fixed-length and the packed problem (the problem statement of "Flash Attention 4":
O = softmax(scale * Q K^T) V with preallocated outputs). The Python binding routes
its calls through the more general fa_fwd_kv / fa_fwd_varlen_kv, so these tests
call the two symbols themselves and compare every element with the fp64 oracle
(O <= 2e-2, LSE <= 1e-3 max-abs, bf16 inputs).
"""
import ctypes
import math

import numpy as np
import pytest

import attention_forward_tma_gb300 as fa
import fa_inputs
import oracle

pytestmark = pytest.mark.gpu

TOL_O = 2e-2
TOL_LSE = 1e-3


@pytest.fixture(scope="module", autouse=True)
def cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.library()
    yield torch


def dev(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def stream():
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def outputs(o, lse):
    import torch
    st, word = fa.last_device_status()
    assert st == fa.FA_OK, hex(word)
    o64 = fa_inputs.bf16_bits_to_f32(o.view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)
    return o64, lse.cpu().numpy().astype(np.float64)


def check(o, lse, o_ref, lse_ref, what):
    assert np.isfinite(o).all(), what
    assert np.abs(o - o_ref).max() <= TOL_O, what
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse), fin), what
    assert np.abs(lse[fin] - lse_ref[fin]).max() <= TOL_LSE, what


@pytest.mark.parametrize("name", ["c1_b1h1n256d64", "c2_b2h8n1024d128"])
@pytest.mark.parametrize("causal", [False, True])
def test_fa_fwd_symbol_against_oracle(name, causal):
    import torch
    w = fa_inputs.WORKLOADS[name]
    x = fa_inputs.make_workload(w)
    q, k, v = dev(x["q"]), dev(x["k"]), dev(x["v"])
    o = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((w.B, w.H, w.N), float("nan"), dtype=torch.float32, device="cuda")
    st = fa.library().fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), w.B, w.H, w.N,
                             w.d, ctypes.c_float(w.scale), int(causal), stream())
    assert st == fa.FA_OK, fa.error_string(st)
    o64, l64 = outputs(o, lse)
    o_ref, l_ref = oracle.attention(x["q"], x["k"], x["v"], w.scale, causal)
    check(o64, l64, o_ref, l_ref, f"fa_fwd {name} causal={causal}")


def test_fa_fwd_symbol_without_lse():
    import torch
    w = fa_inputs.WORKLOADS["c2_b2h8n1024d128"]
    x = fa_inputs.make_workload(w)
    q, k, v = dev(x["q"]), dev(x["k"]), dev(x["v"])
    o = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    st = fa.library().fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), None, w.B, w.H, w.N, w.d,
                             ctypes.c_float(w.scale), 0, stream())
    assert st == fa.FA_OK, fa.error_string(st)
    o64, _ = outputs(o, torch.zeros(1))
    o_ref, _ = oracle.attention(x["q"], x["k"], x["v"], w.scale, False)
    assert np.abs(o64 - o_ref).max() <= TOL_O


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("lengths,H,d", [([700, 0, 129, 1000, 5, 256], 4, 128), ([300, 1, 513], 2, 64)], ids=str)
def test_fa_fwd_varlen_symbol_against_oracle(lengths, H, d, causal):
    import torch
    _, cu, qb, kb, vb = fa_inputs.make_varlen_from_lengths(lengths, H, d, 4000 + sum(lengths))
    T = int(cu[-1])
    q, k, v = dev(qb), dev(kb), dev(vb)
    cu_d = torch.from_numpy(cu).cuda()
    o = torch.full((T, H, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((H, T), float("nan"), dtype=torch.float32, device="cuda")
    scale = 1.0 / math.sqrt(d)
    st = fa.library().fa_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                    cu_d.data_ptr(), len(lengths), T, max(lengths), H, d, ctypes.c_float(scale),
                                    int(causal), stream())
    assert st == fa.FA_OK, fa.error_string(st)
    o64, l64 = outputs(o, lse)
    o_ref, l_ref = oracle.attention_varlen(qb, kb, vb, cu, scale, causal)
    check(o64, l64, o_ref, l_ref, f"fa_fwd_varlen {lengths} causal={causal}")
