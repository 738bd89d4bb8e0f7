"""Pins for the backward oracle (CPU only).

The gradients are tied to things other than their own formulas: central finite
differences of the fp64 forward, PyTorch's float64 autograd of SDPA (an
independent library implementation), and closed forms of the softmax gradient.
The fp64 forward used for the finite differences is itself tied to the C oracle.
"""
import math

import numpy as np
import pytest

import fa_inputs
import oracle


def rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def rand_bits(shape, seed, dtype="bf16"):
    return fa_inputs.f32_to_bits(rand(shape, seed).astype(np.float32), dtype)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dims", [(2, 4, 2, 33, 33, 16), (1, 2, 2, 20, 47, 8), (1, 2, 1, 30, 12, 8)],
                         ids=lambda t: "B%dH%dKV%dNq%dNk%dd%d" % t)
def test_fp64_forward_equals_the_c_oracle(dims, causal):
    B, H, Hkv, Nq, Nk, d = dims
    q = rand_bits((B, Nq, H, d), 1)
    k, v = rand_bits((B, Nk, Hkv, d), 2), rand_bits((B, Nk, Hkv, d), 3)
    o_ref, _ = oracle.attention(q, k, v, 0.3, causal)
    np.testing.assert_allclose(oracle.attention_forward(q, k, v, 0.3, causal), o_ref, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dims", [(1, 2, 1, 4, 6, 3), (1, 2, 2, 5, 5, 2), (1, 1, 1, 6, 3, 2)],
                         ids=lambda t: "B%dH%dKV%dNq%dNk%dd%d" % t)
def test_gradients_match_central_finite_differences(dims, causal):
    """L = sum(dO * O): every input element perturbed by +-h (h = 1e-5); the
    central difference has error O(h^2) ~ 1e-10 relative."""
    B, H, Hkv, Nq, Nk, d = dims
    q, k, v = rand((B, Nq, H, d), 10), rand((B, Nk, Hkv, d), 11), rand((B, Nk, Hkv, d), 12)
    do = rand((B, Nq, H, d), 13)
    s = 0.7
    dq, dk, dv = oracle.attention_backward(q, k, v, do, s, causal)
    h = 1e-5

    def loss(q_, k_, v_):
        return float((do * oracle.attention_forward(q_, k_, v_, s, causal)).sum())

    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            num[idx] = (loss(**{k_ + "_": a for k_, a in args_p.items()}) -
                        loss(**{k_ + "_": a for k_, a in args_m.items()})) / (2 * h)
        np.testing.assert_allclose(g, num, rtol=0, atol=1e-8 * max(1.0, np.abs(num).max()), err_msg=name)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_gradients_match_float64_autograd(causal, dtype):
    torch = pytest.importorskip("torch")
    B, H, Hkv, Nq, Nk, d = 2, 4, 2, 37, 50, 16
    q = rand_bits((B, Nq, H, d), 20, dtype)
    k, v = rand_bits((B, Nk, Hkv, d), 21, dtype), rand_bits((B, Nk, Hkv, d), 22, dtype)
    do = rand_bits((B, Nq, H, d), 23, dtype)
    s = 1.0 / math.sqrt(d)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, s, causal, dtype=dtype)
    t = lambda b: torch.from_numpy(fa_inputs.bits_to_f32(b, dtype).astype(np.float64)).permute(0, 2, 1, 3)  # noqa: E731
    tq, tk, tv = (t(x).requires_grad_() for x in (q, k, v))
    mask = None
    if causal:   # bottom-right alignment: query i sees key j <= i + Nk - Nq
        mask = torch.arange(Nk)[None, :] <= torch.arange(Nq)[:, None] + (Nk - Nq)
    out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=s, enable_gqa=True)
    out.backward(t(do))
    for g, tg in ((dq, tq), (dk, tk), (dv, tv)):
        np.testing.assert_allclose(g, tg.grad.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-12)


def test_closed_forms():
    B, H, N, d = 1, 3, 17, 8
    q, k, v, do = rand((B, N, H, d), 30), rand((B, N, H, d), 31), rand((B, N, H, d), 32), rand((B, N, H, d), 33)
    for causal in (False, True):
        dq, dk, dv = oracle.attention_backward(q, k, v, do, 0.5, causal)
        # every row's weights sum to one: the keys' dV rows sum to the queries' dO rows
        np.testing.assert_allclose(dv.sum(axis=1), do.sum(axis=1), rtol=0, atol=1e-12)
        # shifting every key by one vector adds a per-row constant to the scores: nothing changes
        dq2, dk2, dv2 = oracle.attention_backward(q, k + rand((1, 1, H, d), 34), v, do, 0.5, causal)
        for a, b_ in ((dq, dq2), (dk, dk2), (dv, dv2)):
            np.testing.assert_allclose(a, b_, rtol=0, atol=1e-11)
    # a single key: its weight is 1 for every query, so dQ = dK = 0 and dV = sum of dO
    dq, dk, dv = oracle.attention_backward(q, k[:, :1], v[:, :1], do, 0.5, False)
    assert np.abs(dq).max() < 1e-13 and np.abs(dk).max() < 1e-12
    np.testing.assert_allclose(dv[:, 0], do.sum(axis=1), rtol=0, atol=1e-12)


def test_rows_without_keys_have_no_gradient():
    # causal with Nq > Nk: query rows 0..Nq-Nk-1 see no key (O = 0): dQ there is 0
    q, k, v, do = rand((1, 7, 2, 4), 40), rand((1, 3, 2, 4), 41), rand((1, 3, 2, 4), 42), rand((1, 7, 2, 4), 43)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, 0.5, True)
    assert (dq[:, :4] == 0).all()
    dq2, dk2, dv2 = oracle.attention_backward(q[:, 4:], k, v, do[:, 4:], 0.5, True)
    np.testing.assert_allclose(dk, dk2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(dv, dv2, rtol=0, atol=1e-13)


def test_varlen_with_equal_lengths_is_the_batched_gradient():
    B, H, Hkv, N, d = 3, 4, 2, 9, 8
    q, do = rand((B * N, H, d), 50), rand((B * N, H, d), 51)
    k, v = rand((B * N, Hkv, d), 52), rand((B * N, Hkv, d), 53)
    cu = np.arange(B + 1) * N
    for causal in (False, True):
        got = oracle.attention_backward_varlen(q, k, v, do, cu, cu, 0.4, causal)
        ref = oracle.attention_backward(q.reshape(B, N, H, d), k.reshape(B, N, Hkv, d), v.reshape(B, N, Hkv, d),
                                        do.reshape(B, N, H, d), 0.4, causal)
        for g, r in zip(got, ref):
            np.testing.assert_allclose(g, r.reshape(g.shape), rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_matches_float64_autograd_with_a_block_diagonal_mask(causal):
    """The packed sequences as one attention with a block-diagonal mask (bottom-right
    causal inside each block), differentiated by PyTorch's float64 autograd."""
    torch = pytest.importorskip("torch")
    lq, lk = [3, 5, 2], [4, 5, 6]   # every query row sees at least one key
    H, Hkv, d = 2, 1, 8
    cu_q, cu_k = np.concatenate([[0], np.cumsum(lq)]), np.concatenate([[0], np.cumsum(lk)])
    T, Tk = cu_q[-1], cu_k[-1]
    q, do = rand((T, H, d), 60), rand((T, H, d), 61)
    k, v = rand((Tk, Hkv, d), 62), rand((Tk, Hkv, d), 63)
    dq, dk, dv = oracle.attention_backward_varlen(q, k, v, do, cu_q, cu_k, 0.3, causal)
    mask = torch.zeros(T, Tk, dtype=torch.bool)
    for s in range(len(lq)):
        i = torch.arange(lq[s])[:, None]
        j = torch.arange(lk[s])[None, :]
        blk = (j <= i + (lk[s] - lq[s])) if causal else torch.ones(lq[s], lk[s], dtype=torch.bool)
        mask[cu_q[s]:cu_q[s + 1], cu_k[s]:cu_k[s + 1]] = blk
    t = lambda a: torch.from_numpy(a).permute(1, 0, 2)[None]  # noqa: E731  [1, H, T, d]
    tq, tk, tv = (t(x).clone().requires_grad_() for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=0.3, enable_gqa=True)
    out.backward(t(do))
    for g, tg in ((dq, tq), (dk, tk), (dv, tv)):
        np.testing.assert_allclose(g, tg.grad[0].permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def test_varlen_empty_sequences_and_no_cross_talk():
    lq, lk = [3, 0, 4, 2], [2, 3, 0, 5]
    cu_q, cu_k = np.concatenate([[0], np.cumsum(lq)]), np.concatenate([[0], np.cumsum(lk)])
    q, do = rand((9, 2, 4), 70), rand((9, 2, 4), 71)
    k, v = rand((10, 2, 4), 72), rand((10, 2, 4), 73)
    dq, dk, dv = oracle.attention_backward_varlen(q, k, v, do, cu_q, cu_k, 0.5, False)
    assert (dq[3:7] == 0).all()              # sequence 2 has no keys
    assert (dk[2:5] == 0).all() and (dv[2:5] == 0).all()   # sequence 1 has no queries
    # changing the last sequence's inputs leaves the first sequence's gradients alone
    q2, k2 = q.copy(), k.copy()
    q2[7:] += 1.0
    k2[5:] -= 2.0
    dq2, dk2, dv2 = oracle.attention_backward_varlen(q2, k2, v, do, cu_q, cu_k, 0.5, False)
    assert np.array_equal(dq[:3], dq2[:3]) and np.array_equal(dk[:2], dk2[:2]) and np.array_equal(dv[:2], dv2[:2])
