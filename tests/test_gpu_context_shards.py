"""Key shards of one sequence (fa_fwd_kv_partial) merged through the LSE (fa_lse_combine).

The ranks of a context-sharded call each run fa_fwd_kv_partial on their own key range
and the owner merges the partials ("FlashAttention：一次前向计算", the two-round
example: results over key blocks brought to one reference and divided once by the total
denominator). Here the shards run one after another on one GPU and are merged there, so
everything but the transport is the GPU path; the transport (a gather over
torch.distributed) is tested on CPU ranks in test_dist.py.

Checks: each shard's partial against the oracle over the shard's keys with the whole
sequence's causal diagonal (the oracle's explicit offset), and the merge against the
oracle over all keys, element by element (O <= 2e-2 after the 16-bit merge output;
partial O in fp32 <= 1e-2; LSE <= 1e-3).
"""
import math

import numpy as np
import pytest

import attention_forward_tma_gb300 as fa
import fa_inputs
import oracle
from attention_forward_tma_gb300 import context

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.library()
    yield torch


def dev(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def lse_close(a, b, tol):
    fin = np.isfinite(b)
    assert np.array_equal(np.isfinite(a), fin)
    return (np.abs(a[fin] - b[fin]).max() if fin.any() else 0.0) <= tol


CASES = [  # B, H, H_kv, N_q, N_kv, d, shard sizes
    (2, 4, 2, 1000, 1000, 128, [300, 450, 250]),
    (1, 8, 8, 700, 700, 64, [129, 1, 570]),
    (1, 32, 8, 64, 4096, 128, [1024, 1024, 1024, 1024]),    # decoding-like: few queries, long keys
    (2, 2, 1, 300, 900, 128, [900]),                        # one shard: the whole sequence
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%dH%dKV%dNq%dNk%dd%d_%dshards" % (c[:6] + (len(c[6]),)))
def test_shards_then_merge_against_the_oracle(case, causal):
    import torch
    B, H, Hkv, Nq, Nk, d, sizes = case
    assert sum(sizes) == Nk
    q, k, v = fa_inputs.make_qkv(B, Nq, H, d, seed=900 + Nq + Nk, Nkv=Nk, Hkv=Hkv)
    scale = 1 / math.sqrt(d)
    qd, kd, vd = dev(q), dev(k), dev(v)
    o_parts = torch.full((len(sizes), B, Nq, H, d), float("nan"), dtype=torch.float32, device="cuda")
    lse_parts = torch.full((len(sizes), B, H, Nq), float("nan"), dtype=torch.float32, device="cuda")
    lo = 0
    for i, n in enumerate(sizes):
        fa.fa_fwd_kv_partial(qd, kd[:, lo:lo + n].contiguous(), vd[:, lo:lo + n].contiguous(), lo, Nk,
                             scale=scale, causal=causal, o_part=o_parts[i], lse_part=lse_parts[i])
        lo += n
    o, lse = fa.lse_combine(o_parts, lse_parts)
    st, word = fa.last_device_status()
    assert st == fa.FA_OK, hex(word)
    # each partial against the oracle over its own keys, global diagonal
    lo = 0
    for i, n in enumerate(sizes):
        o_ref, l_ref = oracle.attention(q, k[:, lo:lo + n], v[:, lo:lo + n], scale, causal, off=Nk - Nq - lo)
        op, lp = o_parts[i].cpu().numpy().astype(np.float64), lse_parts[i].cpu().numpy().astype(np.float64)
        assert np.isfinite(op).all()
        assert np.abs(op - o_ref).max() <= 1e-2, (i, np.abs(op - o_ref).max())
        assert lse_close(lp, l_ref, 1e-3), i
        lo += n
    # the merge against the oracle over all keys
    o_ref, l_ref = oracle.attention(q, k, v, scale, causal)
    o64 = fa_inputs.bf16_bits_to_f32(o.view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)
    assert np.abs(o64 - o_ref).max() <= 2e-2
    assert lse_close(lse.cpu().numpy().astype(np.float64), l_ref, 1e-3)


def test_context_sharded_call_on_one_rank():
    """fa_fwd_context_sharded with a world of one (gloo process group on this process):
    the partial, the gather to itself and the merge give the full attention."""
    import os
    import socket
    import torch
    import torch.distributed as dist
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=0, world_size=1)
    try:
        B, H, Nq, Nk, d = 1, 4, 200, 200, 128
        q, k, v = fa_inputs.make_qkv(B, Nq, H, d, seed=31, Nkv=Nk)
        # gloo moves CPU tensors: run the GPU partial, then gather its host copy
        o_part, lse_part = fa.fa_fwd_kv_partial(dev(q), dev(k), dev(v), 0, Nk, causal=True)
        o_parts, lse_parts = context.gather_partials(o_part.cpu(), lse_part.cpu(), dst=0)
        o, lse = fa.lse_combine(o_parts.cuda(), lse_parts.cuda())
        assert fa.last_device_status()[0] == fa.FA_OK
        o_ref, l_ref = oracle.attention(q, k, v, 1 / math.sqrt(d), True)
        o64 = fa_inputs.bf16_bits_to_f32(o.view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)
        assert np.abs(o64 - o_ref).max() <= 2e-2
        assert lse_close(lse.cpu().numpy().astype(np.float64), l_ref, 1e-3)
    finally:
        dist.destroy_process_group()
