"""The allocation-free varlen entry point (fa_fwd_varlen_noalloc).

Some callers cannot allocate device memory when they call attention: a server
that gave all GPU memory to its own pool at start-up, or a latency-critical
loop that must not run allocator calls. fa_fwd_varlen_noalloc serves them by
keeping its work-tile list in a fixed array inside the library. These tests
call it through the C ABI (ctypes) on two calls in a row with different
problems, so stale contents of the shared array from the first call cannot leak
into the second, and check each result against the fp64 oracle (O <= 2e-2,
LSE <= 1e-3 max-abs) and, bit for bit, against fa_fwd_varlen, which runs the
same schedule and kernel from a temporary buffer of the stream-ordered
allocator. This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest

import attention_forward_tma_gb300 as fa
import fa_inputs
import oracle

TOL_O = 2e-2
TOL_LSE = 1e-3


def test_noalloc_rejects_problems_beyond_its_fixed_capacity():
    lib = fa.library()
    # 16 heads x (2^21 / 256 + 1) tiles > 131072: refused before any device work
    st = lib.fa_fwd_varlen_noalloc(256, 256, 256, 256, None, 256, 1, 1 << 21, 1 << 21, 16, 128, 0.088, 1, None)
    assert st == fa.FA_ERR_CAPACITY
    assert "scratch" in fa.error_string(st)


def test_noalloc_capacity_counts_one_tile_tasks_when_forced():
    """With one-tile (128-row) tasks forced, 16 heads x (2^20 / 128 + 1) = 131088 tiles
    exceed the array although 16 x (2^20 / 256 + 1) = 65552 would fit: refused."""
    lib = fa.library()
    T = 1 << 20
    assert 16 * (T // 128 + 1) > 131072 >= 16 * (T // 256 + 1)
    fa.set_option("solo_tiles", 1)
    try:
        st = lib.fa_fwd_varlen_noalloc(256, 256, 256, 256, None, 256, 1, T, T, 16, 128, 0.088, 1, None)
    finally:
        fa.set_option("solo_tiles", -1)
    assert st == fa.FA_ERR_CAPACITY


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
    return o.view(torch.int16).cpu().numpy().view(np.uint16), lse.cpu().numpy()


@pytest.mark.gpu
def test_noalloc_matches_oracle_and_allocating_entry_point_on_two_calls():
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
        o_new, l_new = _run(lib.fa_fwd_varlen_noalloc, qd, kd, vd, cud, maxL, H, d, causal)
        o_ref, l_ref = _run(lib.fa_fwd_varlen, qd, kd, vd, cud, maxL, H, d, causal)
        # the same schedule and kernel as the allocating call: the same bits
        assert np.array_equal(o_new, o_ref)
        assert np.array_equal(l_new.view(np.uint32), l_ref.view(np.uint32))
        # and the oracle's values within the forward tolerances
        o_or, l_or = oracle.attention_varlen(q, k, v, cu, 1.0 / d ** 0.5, causal)
        o64 = fa_inputs.bf16_bits_to_f32(o_new).astype(np.float64)
        assert np.isfinite(o64).all()
        assert np.abs(o64 - o_or).max() <= TOL_O
        fin = np.isfinite(l_or)
        assert np.array_equal(np.isfinite(l_new), fin)
        assert np.abs(l_new[fin].astype(np.float64) - l_or[fin]).max() <= TOL_LSE
