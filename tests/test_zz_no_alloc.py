"""The allocation-free varlen entry point (fa_fwd_varlen_noalloc).

Some callers cannot allocate device memory when they call attention: a server
that gave all GPU memory to its own pool at start-up, or a latency-critical
loop that must not run allocator calls. fa_fwd_varlen_noalloc serves them by
keeping its work-tile list in a fixed array inside the library. These tests
call it through the C ABI (ctypes) and check that it returns what
fa_fwd_varlen (which takes a temporary buffer from the stream-ordered
allocator) returns, on two calls in a row with different problems, so stale
contents of the shared array from the first call cannot leak into the second.
This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest

import attention_forward_tma_gb300 as fa
import fa_inputs

TOL_O = 2e-2
TOL_LSE = 1e-3


def test_noalloc_rejects_problems_beyond_its_fixed_capacity():
    lib = fa.library()
    # 16 heads x (2^21 / 256 + 1) tiles > 131072: refused before any device work
    st = lib.fa_fwd_varlen_noalloc(256, 256, 256, 256, None, 256, 1, 1 << 21, 1 << 21, 16, 128, 0.088, 1, None)
    assert st == fa.FA_ERR_CAPACITY
    assert "scratch" in fa.error_string(st)


def _run(entry, q, k, v, cu, maxL, H, d, causal):
    import torch
    T = q.shape[0]
    o = torch.full((T, H, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((H, T), float("nan"), dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = entry(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), cu.data_ptr(),
               cu.numel() - 1, T, maxL, H, d, ctypes.c_float(1.0 / d ** 0.5), int(causal), stream)
    assert st == fa.FA_OK, fa.error_string(st)
    st, word = fa.last_device_status()
    assert st == fa.FA_OK, hex(word)
    o32 = fa_inputs.bf16_bits_to_f32(o.view(torch.int16).cpu().numpy().view(np.uint16))
    return o32.astype(np.float64), lse.cpu().numpy().astype(np.float64)


@pytest.mark.gpu
def test_noalloc_matches_allocating_entry_point_on_two_calls():
    import torch
    assert torch.cuda.is_available()
    lib = fa.library()

    def dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()

    problems = [([700, 0, 129, 1000, 5], 4, 128, True, 91),     # first call
                ([300, 64], 2, 64, False, 92)]                   # second call: different shape and mask
    for lengths, H, d, causal, seed in problems:
        _, cu, q, k, v = fa_inputs.make_varlen_from_lengths(lengths, H, d, seed)
        qd, kd, vd, cud = dev(q), dev(k), dev(v), torch.from_numpy(cu).cuda()
        maxL = max(lengths)
        o_ref, l_ref = _run(lib.fa_fwd_varlen, qd, kd, vd, cud, maxL, H, d, causal)
        o_new, l_new = _run(lib.fa_fwd_varlen_noalloc, qd, kd, vd, cud, maxL, H, d, causal)
        assert np.isfinite(o_new).all()
        assert np.abs(o_new - o_ref).max() <= TOL_O
        fin = np.isfinite(l_ref)
        assert np.array_equal(np.isfinite(l_new), fin)
        assert np.abs(l_new[fin] - l_ref[fin]).max() <= TOL_LSE
