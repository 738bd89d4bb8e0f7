"""GPU parity at the largest sizes the interface takes: tensors of 2^31 elements
(4 GiB per 16-bit tensor, byte offsets past 2^32 and element offsets up to the
32-bit limit), where an index computed in 32 bits would wrap.

* multi-head B = 128, N = 16384, H = 8, d = 128, causal: Q, K, V, O, dO, dQ, dK and
  dV each hold 2^24 rows of 128 elements; the backward's fp32 dQ accumulator holds
  8 GiB;
* grouped B = 1, N = 131072, H = 128, H_kv = 1 (G = 128), causal: Q and O of 2^31
  elements, one key range and two key ranges merged through their LSE (fp32
  partials of 2^32 elements).

The inputs are tiled from seeded row tables (fa_inputs: row r of a tensor is table
row r * 40503 mod 4099), so any row can be rebuilt on the host. The oracle checks
sampled rows (forward) and whole blocks of rows (backward) against the same
tolerances as the other parity tests: O <= 2e-2 and LSE <= 1e-3 max-abs; gradients
<= 2e-2 * max(1, max |oracle|) per tensor. Rows are sampled at the start, at tile and
table-period boundaries and at the very end of each tensor.
"""
import math

import numpy as np
import pytest

import attention_forward_tma_gb300 as fa
import fa_inputs
import oracle

pytestmark = pytest.mark.gpu

TOL_O, TOL_LSE, TOL_GRAD = 2e-2, 1e-3, 2e-2
SEEDS = {"q": 7100, "k": 7101, "v": 7102, "do": 7103}


@pytest.fixture(scope="module", autouse=True)
def cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.library()
    yield torch
    torch.cuda.synchronize()
    fa.release_cached_memory()    # the backward's 8 GiB workspace
    torch.cuda.empty_cache()


@pytest.fixture(scope="module")
def tables():
    return {name: fa_inputs.make_row_table(128, seed) for name, seed in SEEDS.items()}


def rows_of(table, B, N, heads, b, h, n0=0, n1=None):
    """Positions [n0, n1) of head h of batch b of a tiled [B, N, heads, d] tensor, as
    [1, n1 - n0, 1, d] bit patterns."""
    n = np.arange(n0, N if n1 is None else n1, dtype=np.int64)
    return fa_inputs.tiled_rows(table, (b * N + n) * heads + h)[None, :, None, :]


def host(t):
    import torch
    if t.dtype == torch.bfloat16:
        return fa_inputs.bf16_bits_to_f32(t.view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)
    return t.cpu().numpy().astype(np.float64)


def check_rows(o, lse, o_ref, l_ref, what):
    assert np.isfinite(o).all() and np.isfinite(lse).all(), what
    err_o = np.abs(o - o_ref).max()
    err_l = np.abs(lse - l_ref).max()
    assert err_o <= TOL_O, f"{what}: max |O - oracle| = {err_o}"
    assert err_l <= TOL_LSE, f"{what}: max |LSE - oracle| = {err_l}"


def check_grad(got, ref, what):
    assert np.isfinite(got).all(), what
    bound = TOL_GRAD * max(1.0, np.abs(ref).max())
    err = np.abs(got - ref).max()
    assert err <= bound, f"{what}: max |grad - oracle| = {err} > {bound}"


def test_forward_multi_head_2e31_elements(cuda, tables):
    torch = cuda
    B, N, H, d = 128, 16384, 8, 128
    q = fa_inputs.tiled_tensor_cuda(tables["q"], (B, N, H, d))
    k = fa_inputs.tiled_tensor_cuda(tables["k"], (B, N, H, d))
    v = fa_inputs.tiled_tensor_cuda(tables["v"], (B, N, H, d))
    assert q.numel() == 2 ** 31
    o, lse = fa.fa_fwd(q, k, v, causal=True)
    st, word = fa.last_device_status()
    assert st == fa.FA_OK, hex(word)
    ts = np.array([0, 1, 127, 128, 255, 256, 4098, 4099, 8191, 16382, 16383])
    for b, h in ((0, 0), (63, 3), (127, 7)):
        qb, kb, vb = (rows_of(tables[x], B, N, H, b, h) for x in ("q", "k", "v"))
        rows = np.stack([np.zeros_like(ts), np.zeros_like(ts), ts], axis=1)
        o_ref, l_ref = oracle.attention_rows(qb, kb, vb, rows, 1 / math.sqrt(d), True)
        ti = torch.from_numpy(ts).cuda()
        check_rows(host(o[b, ti, h]), host(lse[b, h, ti]), o_ref, l_ref, f"batch {b} head {h}")
    del q, k, v, o, lse
    torch.cuda.empty_cache()


@pytest.mark.parametrize("splits", [1, 2])
def test_forward_grouped_2e31_elements(cuda, tables, splits):
    """Q and O of 2^31 elements; with two key ranges the fp32 partials hold 2^32."""
    torch = cuda
    B, N, H, Hkv, d = 1, 131072, 128, 1, 128
    q = fa_inputs.tiled_tensor_cuda(tables["q"], (B, N, H, d))
    k = fa_inputs.tiled_tensor_cuda(tables["k"], (B, N, Hkv, d))
    v = fa_inputs.tiled_tensor_cuda(tables["v"], (B, N, Hkv, d))
    o, lse = fa.fa_fwd(q, k, v, causal=True, num_splits=splits)
    st, word = fa.last_device_status()
    assert st == fa.FA_OK, hex(word)
    heads = np.array([0, 1, 64, 127])
    hi = torch.from_numpy(heads).cuda()
    kb, vb = rows_of(tables["k"], B, N, Hkv, 0, 0), rows_of(tables["v"], B, N, Hkv, 0, 0)
    for t in (0, 1, 255, 256, 65535, 65536, 131070, 131071):
        # query position t with all its heads, against keys [0, t]: one query row per
        # head whose bottom-right mask sees every key it is given
        qt = fa_inputs.tiled_rows(tables["q"], t * H + np.arange(H))[None, None, :, :]
        rows = np.stack([np.zeros_like(heads), heads, np.zeros_like(heads)], axis=1)
        o_ref, l_ref = oracle.attention_rows(qt, kb[:, :t + 1], vb[:, :t + 1], rows, 1 / math.sqrt(d), True)
        check_rows(host(o[0, t, hi]), host(lse[0, hi, t]), o_ref, l_ref, f"position {t} splits {splits}")
    del q, k, v, o, lse
    torch.cuda.empty_cache()


def test_backward_multi_head_2e31_elements(cuda, tables):
    """Whole blocks of gradients of two (batch, head) pairs, the first and the last in
    memory: dQ of the first and last 2048 positions and dK, dV of the last 2048 keys (which
    only the last 2048 queries see, so the oracle needs no other query rows)."""
    torch = cuda
    B, N, H, d = 128, 16384, 8, 128
    q, k, v, do = (fa_inputs.tiled_tensor_cuda(tables[x], (B, N, H, d)) for x in ("q", "k", "v", "do"))
    o, lse = fa.fa_fwd(q, k, v, causal=True)
    dq, dk, dv = fa.fa_bwd(q, k, v, o, do, lse, causal=True)
    st, word = fa.last_device_status()
    assert st == fa.FA_OK, hex(word)
    del o, lse
    scale, W = 1 / math.sqrt(d), 2048
    for b, h in ((0, 0), (127, 7)):
        kb, vb = rows_of(tables["k"], B, N, H, b, h), rows_of(tables["v"], B, N, H, b, h)
        qt, dot = (rows_of(tables[x], B, N, H, b, h, N - W) for x in ("q", "do"))
        rq, rk, rv = oracle.attention_backward(qt, kb, vb, dot, scale, True)
        check_grad(host(dq[b, N - W:, h]), rq[0, :, 0], f"dQ tail batch {b} head {h}")
        check_grad(host(dk[b, N - W:, h]), rk[0, N - W:, 0], f"dK tail batch {b} head {h}")
        check_grad(host(dv[b, N - W:, h]), rv[0, N - W:, 0], f"dV tail batch {b} head {h}")
        qh, doh = (rows_of(tables[x], B, N, H, b, h, 0, W) for x in ("q", "do"))
        rq, _, _ = oracle.attention_backward(qh, kb[:, :W], vb[:, :W], doh, scale, True)
        check_grad(host(dq[b, :W, h]), rq[0, :, 0], f"dQ head batch {b} head {h}")
    del q, k, v, do, dq, dk, dv
    torch.cuda.empty_cache()


def test_varlen_forward_and_backward_beyond_2e31_elements(cuda, tables):
    """Packed sequences of 131072, 1, 65535 and 300 positions with H = 128, H_kv = 1:
    Q, O, dO and dQ of 3.2 * 10^9 elements (6 GiB each), the LSE [H, T] of 2.5 * 10^7
    entries. Forward rows at both ends of every sequence; backward: dQ of the long
    sequence's last 128 positions, and every gradient of the last sequence in memory."""
    torch = cuda
    lengths = [131072, 1, 65535, 300]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T, H, d = int(cu[-1]), 128, 128
    cu_d = torch.from_numpy(cu).cuda()
    q, do = (fa_inputs.tiled_tensor_cuda(tables[x], (T, H, d)) for x in ("q", "do"))
    k, v = (fa_inputs.tiled_tensor_cuda(tables[x], (T, 1, d)) for x in ("k", "v"))
    assert q.numel() > 2 ** 31
    o, lse = fa.fa_fwd_varlen(q, k, v, cu_d, max(lengths), causal=True)
    st, word = fa.last_device_status()
    assert st == fa.FA_OK, hex(word)
    scale = 1 / math.sqrt(d)
    heads = np.array([0, 127])
    hi = torch.from_numpy(heads).cuda()

    def seq_rows(name, s, p0, p1, heads_of_row):
        """rows [p0, p1) of sequence s, every head, as [1, p1 - p0, heads_of_row, d]"""
        t = cu[s] + np.arange(p0, p1, dtype=np.int64)
        r = t[:, None] * heads_of_row + np.arange(heads_of_row)[None, :]
        return fa_inputs.tiled_rows(tables[name], r)[None]

    for s, L in enumerate(lengths):
        ks, vs = seq_rows("k", s, 0, L, 1), seq_rows("v", s, 0, L, 1)
        for p in sorted({0, L - 1}):
            qt = seq_rows("q", s, p, p + 1, H)
            rows = np.stack([np.zeros_like(heads), heads, np.zeros_like(heads)], axis=1)
            o_ref, l_ref = oracle.attention_rows(qt, ks[:, :p + 1], vs[:, :p + 1], rows, scale, True)
            t = int(cu[s]) + p
            check_rows(host(o[t, hi]), host(lse[hi, t]), o_ref, l_ref, f"sequence {s} position {p}")

    dq, dk, dv = fa.fa_bwd_varlen(q, k, v, o, do, lse, cu_d, max(lengths), causal=True)
    st, word = fa.last_device_status()
    assert st == fa.FA_OK, hex(word)
    del o, lse
    # the long sequence: dQ of its last W positions, head by head (a query head's dQ
    # needs only its own rows and the sequence's keys)
    L, W = lengths[0], 128
    ks, vs = seq_rows("k", 0, 0, L, 1), seq_rows("v", 0, 0, L, 1)
    qt, dot = seq_rows("q", 0, L - W, L, H), seq_rows("do", 0, L - W, L, H)
    for h in heads:
        rq, _, _ = oracle.attention_backward(qt[:, :, h:h + 1], ks, vs, dot[:, :, h:h + 1], scale, True)
        check_grad(host(dq[L - W:L, h]), rq[0, :, 0], f"dQ tail of sequence 0 head {h}")
    # the last sequence: all heads, all gradients
    s = len(lengths) - 1
    a, e = int(cu[s]), int(cu[s + 1])
    ref = oracle.attention_backward(seq_rows("q", s, 0, e - a, H), seq_rows("k", s, 0, e - a, 1),
                                    seq_rows("v", s, 0, e - a, 1), seq_rows("do", s, 0, e - a, H), scale, True)
    for name, got, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        check_grad(host(got[a:e]), r[0], f"{name} of sequence {s}")
    del q, k, v, do, dq, dk, dv
    torch.cuda.synchronize()
    fa.release_cached_memory()
    torch.cuda.empty_cache()
