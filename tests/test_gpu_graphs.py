"""The entry points inside a captured CUDA graph: after one eager call (which sets the
kernels' attributes), a forward, a variable-length forward (its schedule kernel and
task list) and a backward are captured on a stream and replayed; the replays give
the eager results (the forward and dK, dV bit for bit; dQ, summed over key blocks in
arrival order, within the backward's tolerance)."""
import math

import numpy as np
import pytest

import attention_forward_tma_gb300 as fa
import fa_inputs
import oracle

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


def host(t):
    import torch
    if t.dtype == torch.bfloat16:
        return fa_inputs.bf16_bits_to_f32(t.view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)
    return t.cpu().numpy().astype(np.float64)


def test_forward_and_backward_in_a_cuda_graph():
    import torch
    q, k, v = fa_inputs.make_qkv(2, 600, 8, 128, seed=4700, Hkv=2)
    do = fa_inputs.make_qkv(2, 600, 8, 128, seed=4701)[0]
    qd, kd, vd, dod = dev(q), dev(k), dev(v), dev(do)
    lengths = [300, 1, 257, 42]
    _, cu, vq, vk, vv = fa_inputs.make_varlen_from_lengths(lengths, 4, 128, seed=4702, Hkv=2)
    vqd, vkd, vvd, cud = dev(vq), dev(vk), dev(vv), torch.from_numpy(cu).cuda()

    def work():
        o, lse = fa.fa_fwd(qd, kd, vd, causal=True)
        dq, dk, dv = fa.fa_bwd(qd, kd, vd, o, dod, lse, causal=True)
        vo, vlse = fa.fa_fwd_varlen(vqd, vkd, vvd, cud, max(lengths), causal=True)
        return o, lse, dq, dk, dv, vo, vlse

    eager = [t.clone() for t in work()]
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        work()                                   # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        outs = work()
    for _ in range(2):
        for t in outs:
            t.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        st, word = fa.last_device_status()
        assert st == fa.FA_OK, hex(word)
        for i in (0, 1, 3, 4, 5, 6):             # forward outputs, dK, dV: bit for bit
            assert torch.equal(outs[i], eager[i]), i
        ref = oracle.attention_backward(q, k, v, do, 1 / math.sqrt(128), True)
        err = np.abs(host(outs[2]) - ref[0]).max()
        assert err <= 2e-2 * max(1.0, np.abs(ref[0]).max()), err
