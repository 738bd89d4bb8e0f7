"""Device-side checks of cu_seqlens for the packed (varlen) calls.

The varlen design reads each sequence's offsets from cu_seqlens on the device
("FlashAttention-4（下）", section "6. LPT 调度": a pre-kernel reads the sequence
lengths and orders the work tiles). The offsets are device data the host does not
read, so the forward's schedule kernel and a one-block kernel in front of the
backward check them before any other work: cu_seqlens[0] = 0, non-decreasing, the
last entry equal to the packed row count, and every length within the maximum the
caller passed. A broken array makes the call write nothing and
fa_last_device_status report FA_ERR_INVALID_ARG, with role 7 and the first
offending sequence in the detail word. Every array here is built on the host; no
kernel reads past it, so none of these cases touches memory outside the buffers.
"""
import numpy as np
import pytest

import attention_forward_tma_gb300 as fa
import fa_inputs
import oracle

pytestmark = pytest.mark.gpu

LENGTHS = [300, 64, 500]
H, D = 2, 128
T = sum(LENGTHS)
GOOD = [0, 300, 364, 864]
# (name, cu_seqlens, max_seqlen, first offending sequence)
BAD = [
    ("first_entry_not_zero", [4, 300, 364, 864], 500, 0),
    ("decreasing", [0, 300, 200, 864], 700, 1),
    ("last_entry_not_total", [0, 300, 364, 800], 500, 2),
    ("length_above_max_seqlen", GOOD, 400, 2),
]
SENTINEL = 7.0


@pytest.fixture(scope="module")
def inputs():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.library()
    cu = np.array(GOOD, np.int32)
    _, cu_chk, q, k, v = fa_inputs.make_varlen_from_lengths(LENGTHS, H, D, 515)
    assert np.array_equal(cu, cu_chk)

    def dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()

    return {"bits": (q, k, v), "dev": (dev(q), dev(k), dev(v))}


def expect_rejected(first_bad):
    st, word = fa.last_device_status()
    assert st == fa.FA_ERR_INVALID_ARG, (st, hex(word))
    assert (word >> 8) & 0xff == 7 and word >> 32 == first_bad, hex(word)


@pytest.mark.parametrize("splits", [1, 2])
@pytest.mark.parametrize("name,cu,max_len,first_bad", BAD, ids=[b[0] for b in BAD])
def test_forward_rejects_bad_offsets_and_writes_nothing(inputs, name, cu, max_len, first_bad, splits):
    import torch
    q, k, v = inputs["dev"]
    cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
    o = torch.full((T, H, D), SENTINEL, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((H, T), SENTINEL, dtype=torch.float32, device="cuda")
    fa.fa_fwd_varlen(q, k, v, cu_d, max_len, causal=True, out=o, lse=lse, num_splits=splits)
    expect_rejected(first_bad)
    assert bool((o == SENTINEL).all()) and bool((lse == SENTINEL).all())


def test_forward_after_a_rejected_call_is_correct(inputs):
    """The rejection leaves nothing behind: the next call with valid offsets matches the oracle."""
    import torch
    q, k, v = inputs["dev"]
    fa.fa_fwd_varlen(q, k, v, torch.tensor(BAD[1][1], dtype=torch.int32, device="cuda"), 700, causal=True)
    expect_rejected(1)
    o, lse = fa.fa_fwd_varlen(q, k, v, torch.tensor(GOOD, dtype=torch.int32, device="cuda"), max(LENGTHS),
                              causal=True)
    st, word = fa.last_device_status()
    assert st == fa.FA_OK, hex(word)
    o64 = fa_inputs.bf16_bits_to_f32(o.view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)
    qb, kb, vb = inputs["bits"]
    o_ref, l_ref = oracle.attention_varlen(qb, kb, vb, np.array(GOOD, np.int32), 1 / D ** 0.5, True)
    assert np.abs(o64 - o_ref).max() <= 2e-2
    assert np.abs(lse.cpu().numpy() - l_ref).max() <= 1e-3


@pytest.mark.parametrize("name,cu,max_len,first_bad", BAD, ids=[b[0] for b in BAD])
def test_backward_rejects_bad_offsets_and_writes_nothing(inputs, name, cu, max_len, first_bad):
    import torch
    q, k, v = inputs["dev"]
    good = torch.tensor(GOOD, dtype=torch.int32, device="cuda")
    o, lse = fa.fa_fwd_varlen(q, k, v, good, max(LENGTHS), causal=True)
    assert fa.last_device_status()[0] == fa.FA_OK
    dout = torch.ones_like(q)
    grads = [torch.full_like(t, SENTINEL) for t in (q, k, v)]
    fa.fa_bwd_varlen(q, k, v, o, dout, lse, torch.tensor(cu, dtype=torch.int32, device="cuda"), max_len,
                     causal=True, dq=grads[0], dk=grads[1], dv=grads[2])
    expect_rejected(first_bad)
    for g in grads:
        assert bool((g == SENTINEL).all())
