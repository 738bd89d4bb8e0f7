"""Solo tasks of the forward: one 128-row Q tile per task, its score tile alternating
between the two S buffers of tensor memory so that a key block's QK^T overlaps the
previous block's softmax, and both softmax warpgroups sharing the tile (64 key columns
each). Every row visits the same key blocks in the same order with the same reference
and the same P, so O and the LSE differ from two-tile tasks only through the row sum's
summation order (two partial sums): at most one 16-bit unit in the last place of O and
1e-5 in the LSE. Both must match the fp64 oracle (O <= 2e-2, LSE <= 1e-3 max-abs).

The shapes cover an even and an odd number of key blocks per task, one block, grouped
heads up to G = 128, N_q != N_kv (causal rows without keys), key splits, decoding, and
spiky scores whose delayed rescale makes the correction warpgroup wait for the previous
block's PV (the statistics through tensor memory and through shared memory).
"""
import math

import numpy as np
import pytest

import attention_forward_tma_gb300 as fa
import fa_inputs
import oracle

pytestmark = pytest.mark.gpu

TOL_O, TOL_LSE = 2e-2, 1e-3


@pytest.fixture(scope="module", autouse=True)
def cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.library()
    yield torch
    fa.set_option("solo_tiles", -1)
    fa.set_option("stats_tmem", 1)


def dev(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def host(t):
    import torch
    if t.dtype == torch.bfloat16:
        return fa_inputs.bf16_bits_to_f32(t.view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)
    return t.cpu().numpy().astype(np.float64)


def run(q, k, v, causal, splits, solo, stats_tmem=1):
    fa.set_option("solo_tiles", solo)
    fa.set_option("stats_tmem", stats_tmem)
    try:
        o, lse = fa.fa_fwd(dev(q), dev(k), dev(v), causal=causal, num_splits=splits)
        st, word = fa.last_device_status()
    finally:
        fa.set_option("solo_tiles", -1)
        fa.set_option("stats_tmem", 1)
    assert st == fa.FA_OK, hex(word)
    return host(o), host(lse)


def same_up_to_row_sum_order(a, b, what):
    """O within one bf16 unit in the last place (2^-7 relative) plus 1e-5 absolute (an
    output merged from key ranges can cancel to near zero while the ranges' own rounding
    is relative to their larger partial outputs), LSE within 1e-5."""
    bad = np.abs(a[0] - b[0]) > 2.0 ** -7 * np.abs(b[0]) + 1e-5
    if bad.any():
        idx = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: O differs at {int(bad.sum())} elements, first {idx}: "
                             f"{a[0][idx]} against {b[0][idx]}")
    fin = np.isfinite(b[1])
    assert (np.isfinite(a[1]) == fin).all(), what
    assert np.abs(a[1][fin] - b[1][fin]).max(initial=0.0) <= 1e-5, f"{what}: LSE differs"


def check(o, lse, o_ref, l_ref, what):
    assert np.isfinite(o).all(), what
    err_o = np.abs(o - o_ref).max()
    assert err_o <= TOL_O, f"{what}: max |O - oracle| = {err_o}"
    fin = np.isfinite(l_ref)
    assert (np.isneginf(lse) == ~fin).all(), what
    err_l = np.abs(lse[fin] - l_ref[fin]).max() if fin.any() else 0.0
    assert err_l <= TOL_LSE, f"{what}: max |LSE - oracle| = {err_l}"


SHAPES = [  # (B, H, H_kv, N_q, N_kv, d, splits)
    (1, 2, 2, 1100, 1100, 128, 1),    # 9 key blocks: odd count
    (2, 3, 3, 700, 700, 64, 1),       # 6 key blocks: even count
    (1, 2, 2, 100, 100, 128, 1),      # one key block
    (1, 8, 2, 300, 300, 128, 1),      # G = 4
    (1, 128, 1, 40, 300, 64, 1),      # G = 128: one position per tile
    (1, 4, 1, 200, 650, 128, 1),      # N_q < N_kv
    (1, 2, 2, 650, 200, 128, 1),      # N_q > N_kv: causal rows without keys
    (1, 4, 2, 500, 1500, 128, 3),     # key ranges merged through their LSE
    (2, 32, 8, 1, 4096, 128, 0),      # decoding, the library's key ranges
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%dH%dKV%dNq%dNk%dd%ds%d" % s)
def test_solo_matches_two_tile_tasks_and_oracle(shape, causal):
    B, H, Hkv, Nq, Nk, d, splits = shape
    q, k, v = fa_inputs.make_qkv(B, Nq, H, d, seed=8000 + Nq + Nk + H, Nkv=Nk, Hkv=Hkv)
    solo = run(q, k, v, causal, splits, 1)
    two = run(q, k, v, causal, splits, 0)
    same_up_to_row_sum_order(solo, two, f"{shape} causal={causal}")
    o_ref, l_ref = oracle.attention(q, k, v, 1 / math.sqrt(d), causal)
    check(solo[0], solo[1], o_ref, l_ref, f"{shape} causal={causal}")


@pytest.mark.parametrize("stats_tmem", [1, 0])
def test_solo_rescales_wait_for_the_previous_pv(stats_tmem):
    """Spiky scores: row references move by more than tau, so the correction warpgroup
    rescales O, which in a solo task first waits for the previous block's PV."""
    q, k, v = fa_inputs.make_qkv(1, 1500, 4, 128, seed=20264, spiky=True)
    solo = run(q, k, v, True, 1, 1, stats_tmem)
    two = run(q, k, v, True, 1, 0, stats_tmem)
    same_up_to_row_sum_order(solo, two, f"spiky stats_tmem={stats_tmem}")
    o_ref, l_ref = oracle.attention(q, k, v, 1 / math.sqrt(128), True)
    check(solo[0], solo[1], o_ref, l_ref, f"spiky stats_tmem={stats_tmem}")


@pytest.mark.parametrize("shape", [(4, 32, 8, 1, 16384), (2, 8, 8, 1024, 1024), (1, 32, 8, 1, 4096)],
                         ids=lambda s: "B%dH%dKV%dNq%dNk%d" % s)
def test_split_query_matches_the_call(shape):
    """fa_fwd_kv_splits reports the key ranges a num_splits=0 call uses (with the task
    size the library picks): the call with that count given explicitly is bit-identical."""
    import torch
    B, H, Hkv, Nq, Nk = shape
    q, k, v = fa_inputs.make_qkv(B, Nq, H, 128, seed=8100 + B + Nq, Nkv=Nk, Hkv=Hkv)
    qd, kd, vd = dev(q), dev(k), dev(v)
    n = fa.num_splits(B, H, Hkv, Nq, Nk, 0, causal=True, d=128)
    a = fa.fa_fwd(qd, kd, vd, causal=True, num_splits=0)
    b = fa.fa_fwd(qd, kd, vd, causal=True, num_splits=n)
    st, word = fa.last_device_status()
    assert st == fa.FA_OK, hex(word)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("d", [64, 128])
def test_solo_fp16(d):
    """fp16 inputs through the solo kernel (P in fp16, tau capped at 15), grouped heads."""
    import torch
    q, k, v = fa_inputs.make_qkv(1, 333, 8, d, seed=8200 + d, Hkv=2, dtype="f16")
    to = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.float16).cuda()
    out = {}
    for solo in (1, 0):
        fa.set_option("solo_tiles", solo)
        try:
            o, lse = fa.fa_fwd(to(q), to(k), to(v), causal=True)
            st, word = fa.last_device_status()
        finally:
            fa.set_option("solo_tiles", -1)
        assert st == fa.FA_OK, hex(word)
        out[solo] = (o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64))
    same_up_to_row_sum_order(out[1], out[0], f"fp16 d={d}")
    o_ref, l_ref = oracle.attention(q, k, v, 1 / math.sqrt(d), True, dtype="f16")
    check(out[1][0], out[1][1], o_ref, l_ref, f"fp16 d={d}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("lq,lk", [([7, 0, 129, 300, 1, 520], None), ([1, 1, 1, 1], [700, 1, 129, 4096])],
                         ids=["self", "decode"])
def test_solo_varlen(lq, lk, causal):
    """Packed batches through solo tasks (the schedule kernel cuts 128-row tiles):
    self-attention with empty and one-row sequences, and decoding (one query row per
    sequence against its own key length), against two-tile tasks and the oracle."""
    import torch
    H, Hkv, d = 8, 2, 128
    lk = lq if lk is None else lk
    rng = np.random.default_rng(sum(lq) + 3 * sum(lk))
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    q = fa_inputs.f32_to_bits(rng.standard_normal((int(cu_q[-1]), H, d), dtype=np.float32), "bf16")
    k = fa_inputs.f32_to_bits(rng.standard_normal((int(cu_k[-1]), Hkv, d), dtype=np.float32), "bf16")
    v = fa_inputs.f32_to_bits(rng.standard_normal((int(cu_k[-1]), Hkv, d), dtype=np.float32), "bf16")
    cq, ck = torch.from_numpy(cu_q).cuda(), torch.from_numpy(cu_k).cuda()
    out = {}
    for solo in (1, 0):
        fa.set_option("solo_tiles", solo)
        try:
            o, lse = fa.fa_fwd_varlen(dev(q), dev(k), dev(v), cq, max(lq), causal=causal, cu_seqlens_k=ck,
                                      max_seqlen_k=max(lk), num_splits=0)
            st, word = fa.last_device_status()
        finally:
            fa.set_option("solo_tiles", -1)
        assert st == fa.FA_OK, hex(word)
        out[solo] = (host(o), host(lse))
    same_up_to_row_sum_order(out[1], out[0], f"varlen {lq} {lk}")
    o_ref = np.zeros((int(cu_q[-1]), H, d))
    l_ref = np.full((H, int(cu_q[-1])), -np.inf)
    for s in range(len(lq)):
        a, b, c, e = int(cu_q[s]), int(cu_q[s + 1]), int(cu_k[s]), int(cu_k[s + 1])
        if b == a:
            continue
        os_, ls_ = oracle.attention(q[None, a:b], k[None, c:e], v[None, c:e], 1 / math.sqrt(d), causal)
        o_ref[a:b] = os_[0]
        l_ref[:, a:b] = ls_[0]
    check(out[1][0], out[1][1], o_ref, l_ref, f"varlen {lq} {lk} causal={causal}")
