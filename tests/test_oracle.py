"""Pins for the fp64 oracle (CPU only).

Each check ties the oracle to something other than itself: values printed on
the pages (fixtures in tests/golden, each citing its page and figure), closed
forms of softmax attention, exact-rational brute force on tiny inputs, and the
float64 SDPA routine of PyTorch as an independent library implementation.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import fa_inputs
import oracle
from tests.golden import fixtures

LN2 = math.log(2.0)


def bits(x):
    a = np.asarray(x, dtype=np.float32)
    b = fa_inputs.f32_to_bf16_bits(a)
    assert np.array_equal(fa_inputs.bf16_bits_to_f32(b), a), "fixture values must be exact in bf16"
    return b


def as_float(rows):
    return np.array([[float(x) for x in r] for r in rows], dtype=np.float64)


def one_head(x):
    """[N, d] -> [1, N, 1, d]"""
    return np.asarray(x)[None, :, None, :]


# --------------------------------------------------------------------------- pages
def test_p3_two_round_example_final_values():
    g = fixtures.load("p3_two_round_example.txt")
    q, k, v = (bits(as_float(g[n])) for n in ("Q", "K", "V"))
    o, lse = oracle.attention(one_head(q), one_head(k), one_head(v), scale=LN2, causal=False)
    np.testing.assert_allclose(o[0, :, 0, :], as_float(g["O"]), rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], [math.log(float(x)) for x in g["LSE_ln"]], rtol=0, atol=1e-14)
    # the printed score matrix: S = Q K^T before the scale
    np.testing.assert_array_equal(as_float(g["Q"]) @ as_float(g["K"]).T, as_float(g["S"]))


def test_p3_causal_fig12_top_left_and_bottom_right():
    g = fixtures.load("p3_two_round_example.txt")
    c = fixtures.load("p3_causal_fig12.txt")
    q, k, v = (one_head(bits(as_float(g[n]))) for n in ("Q", "K", "V"))
    o, lse = oracle.attention(q, k, v, scale=LN2, causal=True, off=0)          # top-left
    np.testing.assert_allclose(o[0, :, 0, :], as_float(c["O_TOPLEFT"]), atol=1e-14, rtol=0)
    np.testing.assert_allclose(lse[0, 0], [math.log(float(x)) for x in c["LSE_TOPLEFT_ln"]],
                               atol=1e-14, rtol=0)
    o, lse = oracle.attention(q, k, v, scale=LN2, causal=True)                 # bottom-right
    np.testing.assert_allclose(o[0, :, 0, :], as_float(c["O_BOTTOMRIGHT"]), atol=1e-14, rtol=0)
    np.testing.assert_allclose(lse[0, 0], [math.log(float(x)) for x in c["LSE_BOTTOMRIGHT_ln"]],
                               atol=1e-14, rtol=0)


def test_p1_exercise7_bottom_right_visibility():
    """N_q = 6, N_kv = 8: query i sees exactly keys 0..max_key[i] (one-hot V reveals the set)."""
    ex = fixtures.load("p1_exercises.txt")
    max_key = [int(x) for x in ex["EX7_MAX_KEY"]]
    nq, nkv, d = 6, 8, 8
    q = np.zeros((nq, d), np.float32)             # equal scores: uniform weight on visible keys
    k = np.zeros((nkv, d), np.float32)
    v = np.eye(nkv, d, dtype=np.float32)          # row j of V is the j-th unit vector
    o, lse = oracle.attention(one_head(bits(q)), one_head(bits(k)), one_head(bits(v)),
                              scale=0.125, causal=True)
    for i in range(nq):
        want = np.zeros(d)
        want[: max_key[i] + 1] = 1.0 / (max_key[i] + 1)
        np.testing.assert_allclose(o[0, i, 0], want, atol=1e-15, rtol=0)
        assert lse[0, 0, i] == pytest.approx(math.log(max_key[i] + 1), abs=1e-15)


# --------------------------------------------------------------------------- closed forms
def rand_bits(shape, seed):
    rng = np.random.default_rng(seed)
    return fa_inputs.f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32))


@pytest.mark.parametrize("causal", [False, True])
def test_equal_scores_give_mean_of_v(causal):
    B, N, H, d = 2, 37, 3, 16
    q = np.zeros((B, N, H, d), np.uint16)                       # all scores are 0
    k = rand_bits((B, N, H, d), 1)
    v = rand_bits((B, N, H, d), 2)
    o, lse = oracle.attention(q, k, v, scale=0.3, causal=causal)
    vf = fa_inputs.bf16_bits_to_f32(v).astype(np.float64)
    for i in range(N):
        n = i + 1 if causal else N
        np.testing.assert_allclose(o[:, i], vf[:, :n].mean(axis=1), atol=1e-13, rtol=0)
        np.testing.assert_allclose(lse[:, :, i], math.log(n), atol=1e-13, rtol=0)


def test_constant_v_and_weights_sum_to_one():
    """V = c in every row gives O = c: the softmax weights of every row sum to 1."""
    B, N, H, d = 1, 50, 2, 8
    q = rand_bits((B, N, H, d), 3)
    k = rand_bits((B, N, H, d), 4)
    c = bits(np.arange(-4, 4, dtype=np.float32) / 4)
    v = np.broadcast_to(c, (B, N, H, d)).copy()
    cf = fa_inputs.bf16_bits_to_f32(c).astype(np.float64)
    for causal in (False, True):
        o, _ = oracle.attention(q, k, v, scale=0.25, causal=causal)
        np.testing.assert_allclose(o, np.broadcast_to(cf, o.shape), atol=1e-13, rtol=0)


def test_dominant_key_returns_its_value_row():
    N, d, j = 40, 16, 17
    rng = np.random.default_rng(5)
    qf = rng.standard_normal((N, d)).astype(np.float32)
    kf = (0.05 * rng.standard_normal((N, d))).astype(np.float32)
    kf[j] = 1.0                                            # q.k_j >> q.k_other for q = all-ones
    qf[:] = 1.0
    q = bits(qf)
    k = fa_inputs.f32_to_bf16_bits(kf)
    v = rand_bits((N, d), 6)
    scale = 4.0
    o, lse = oracle.attention(one_head(q), one_head(k), one_head(v), scale=scale, causal=False)
    vf = fa_inputs.bf16_bits_to_f32(v).astype(np.float64)
    # every other weight is below exp(-scale*(16 - 16*0.05*4)) relative to the dominant one
    np.testing.assert_allclose(o[0, :, 0], np.broadcast_to(vf[j], (N, d)), atol=1e-12, rtol=0)
    kd = fa_inputs.bf16_bits_to_f32(k).astype(np.float64)
    np.testing.assert_allclose(lse[0, 0], scale * kd[j].sum(), atol=1e-12, rtol=0)


def test_causal_row_zero_is_first_value_row():
    B, N, H, d = 2, 33, 2, 8
    q, k, v = rand_bits((B, N, H, d), 7), rand_bits((B, N, H, d), 8), rand_bits((B, N, H, d), 9)
    o, lse = oracle.attention(q, k, v, scale=0.5, causal=True)
    vf = fa_inputs.bf16_bits_to_f32(v).astype(np.float64)
    qf = fa_inputs.bf16_bits_to_f32(q).astype(np.float64)
    kf = fa_inputs.bf16_bits_to_f32(k).astype(np.float64)
    np.testing.assert_array_equal(o[:, 0], vf[:, 0])
    np.testing.assert_allclose(lse[:, :, 0], 0.5 * np.einsum("bhd,bhd->bh", qf[:, 0], kf[:, 0]),
                               atol=1e-13, rtol=0)


def test_linear_in_v_and_permutation_invariant():
    B, N, H, d = 1, 29, 2, 8
    q, k = rand_bits((B, N, H, d), 10), rand_bits((B, N, H, d), 11)
    v1, v2 = rand_bits((B, N, H, d), 12), rand_bits((B, N, H, d), 13)
    f = lambda b: fa_inputs.bf16_bits_to_f32(b).astype(np.float64)  # noqa: E731
    # scaling V by 2 is exact in bf16, so O must scale by exactly 2
    o1, _ = oracle.attention(q, k, v1, 0.4, False)
    o2, _ = oracle.attention(q, k, v2, 0.4, False)
    o12, _ = oracle.attention(q, k, fa_inputs.f32_to_bf16_bits(f(v1).astype(np.float32) * 2), 0.4, False)
    np.testing.assert_allclose(o12, 2 * o1, atol=1e-13, rtol=0)
    # linearity of a sum: use V columns drawn so that v1 + v2 stays exact (disjoint supports)
    va = v1.copy(); va[..., d // 2:] = 0
    vb = v2.copy(); vb[..., : d // 2] = 0
    oa, _ = oracle.attention(q, k, va, 0.4, False)
    ob, _ = oracle.attention(q, k, vb, 0.4, False)
    oab, _ = oracle.attention(q, k, va | vb, 0.4, False)
    np.testing.assert_allclose(oab, oa + ob, atol=1e-13, rtol=0)
    # joint permutation of the K and V rows leaves the non-causal output unchanged
    perm = np.random.default_rng(14).permutation(N)
    op, lp = oracle.attention(q, k[:, perm], v1[:, perm], 0.4, False)
    o0, l0 = oracle.attention(q, k, v1, 0.4, False)
    np.testing.assert_allclose(op, o0, atol=1e-13, rtol=0)
    np.testing.assert_allclose(lp, l0, atol=1e-13, rtol=0)


def test_empty_rows_give_zero_and_minus_inf():
    """Rows with no visible key (possible only with N_q > N_kv) -> O = 0, LSE = -inf."""
    q, k, v = rand_bits((1, 6, 1, 4), 15), rand_bits((1, 3, 1, 4), 16), rand_bits((1, 3, 1, 4), 17)
    o, lse = oracle.attention(q, k, v, 0.5, True)             # off = -3: rows 0..2 see nothing
    assert np.all(o[0, :3] == 0) and np.all(np.isneginf(lse[0, 0, :3]))
    assert np.all(np.isfinite(lse[0, 0, 3:]))


# --------------------------------------------------------------------------- brute force
def exact_attention(qi, ki, vi, causal, off):
    """Exact rationals: s = ln 2 and integer scores make every weight a power of two."""
    nq, nkv = len(qi), len(ki)
    O, L = [], []
    for i in range(nq):
        valid = [j for j in range(nkv) if (not causal) or j <= i + off]
        t = {j: sum(a * b for a, b in zip(qi[i], ki[j])) for j in valid}
        m = max(t.values())
        w = {j: Fraction(2) ** (t[j] - m) for j in valid}
        den = sum(w.values())
        O.append([sum(w[j] * vi[j][c] for j in valid) / den for c in range(len(vi[0]))])
        L.append(m * LN2 + math.log(den))
    return O, L


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_exact_rationals(seed):
    rng = np.random.default_rng(100 + seed)
    nq = int(rng.integers(1, 8))
    nkv = int(rng.integers(nq, 9))
    d = int(rng.integers(1, 5))
    causal = bool(seed % 2)
    qi = rng.integers(-2, 3, (nq, d)).tolist()
    ki = rng.integers(-2, 3, (nkv, d)).tolist()
    vi = rng.integers(-4, 5, (nkv, d)).tolist()
    O, L = exact_attention(qi, ki, vi, causal, nkv - nq)
    q, k, v = (one_head(bits(np.array(x, np.float32))) for x in (qi, ki, vi))
    o, lse = oracle.attention(q, k, v, scale=LN2, causal=causal)
    np.testing.assert_allclose(o[0, :, 0], np.array([[float(x) for x in r] for r in O]),
                               atol=1e-13, rtol=0)
    np.testing.assert_allclose(lse[0, 0], L, atol=1e-13, rtol=0)


# --------------------------------------------------------------------------- library routine
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(2, 3, 70, 64), (1, 2, 129, 128), (1, 1, 1, 64)])
def test_matches_float64_sdpa(shape, causal):
    torch = pytest.importorskip("torch")
    B, H, N, d = shape
    q, k, v = (rand_bits((B, N, H, d), s) for s in (20, 21, 22))
    scale = 1.0 / math.sqrt(d)
    o, lse = oracle.attention(q, k, v, scale, causal)
    t = lambda b: torch.from_numpy(fa_inputs.bf16_bits_to_f32(b).astype(np.float64)).permute(0, 2, 1, 3)  # noqa: E731
    ref = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), scale=scale, is_causal=causal)
    np.testing.assert_allclose(o, ref.permute(0, 2, 1, 3).numpy(), atol=1e-12, rtol=0)
    s = torch.einsum("bhid,bhjd->bhij", t(q), t(k)) * scale
    if causal:
        s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), atol=1e-12, rtol=0)


# --------------------------------------------------------------------------- entry points agree
def test_varlen_equals_per_sequence_fixed_length():
    lengths = [5, 0, 130, 1, 64]
    H, d = 3, 16
    _, cu, q, k, v = fa_inputs.make_varlen_from_lengths(lengths, H, d, seed=30)
    for causal in (False, True):
        o, lse = oracle.attention_varlen(q, k, v, cu, 0.3, causal)
        for s, L in enumerate(lengths):
            a, b = int(cu[s]), int(cu[s + 1])
            if L == 0:
                continue
            of, lf = oracle.attention(q[None, a:b], k[None, a:b], v[None, a:b], 0.3, causal)
            np.testing.assert_array_equal(o[a:b], of[0])
            np.testing.assert_array_equal(lse[:, a:b], lf[0])


def test_rows_equal_full_result():
    B, N, H, d = 2, 77, 3, 32
    q, k, v = (rand_bits((B, N, H, d), s) for s in (40, 41, 42))
    o, lse = oracle.attention(q, k, v, 0.2, True)
    rows = np.array([[0, 0, 0], [1, 2, 76], [0, 1, 33], [1, 0, 5]], np.int64)
    orow, lrow = oracle.attention_rows(q, k, v, rows, 0.2, True)
    for r, (b, h, i) in enumerate(rows):
        np.testing.assert_array_equal(orow[r], o[b, i, h])
        assert lrow[r] == lse[b, h, i]
    lengths = [7, 0, 90]
    _, cu, q2, k2, v2 = fa_inputs.make_varlen_from_lengths(lengths, 2, 16, seed=43)
    o2, l2 = oracle.attention_varlen(q2, k2, v2, cu, 0.25, True)
    rows2 = np.array([[0, 0], [1, 6], [0, 7], [1, 96]], np.int64)
    orow2, lrow2 = oracle.attention_rows_varlen(q2, k2, v2, cu, rows2, 0.25, True)
    for r, (h, t) in enumerate(rows2):
        np.testing.assert_array_equal(orow2[r], o2[t, h])
        assert lrow2[r] == l2[h, t]


def test_invalid_arguments_raise():
    q = np.zeros((1, 4, 1, 8), np.uint16)
    with pytest.raises(ValueError):
        oracle.attention_rows(q, q, q, np.array([[0, 0, 4]]), 0.5, False)
    with pytest.raises(TypeError):
        oracle.attention(q.astype(np.float32), q, q, 0.5, False)


# --------------------------------------------------------------------------- element types
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_every_16bit_pattern_widens_exactly(dtype):
    """With a single key the weights are exactly 1, so O is V widened to double:
    every one of the 65536 bit patterns (zeros, subnormals, normals, infinities,
    NaNs) must come back as numpy's own widening of that pattern."""
    pat = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = pat.reshape(1, 1, 1, -1)
    z = np.zeros_like(v)
    o, lse = oracle.attention(z, z, v, 0.5, False, dtype=dtype)
    with np.errstate(invalid="ignore"):   # signalling NaN patterns widen to quiet NaNs
        if dtype == "f16":
            want = pat.view(np.float16).astype(np.float64)
        else:
            want = (pat.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    np.testing.assert_array_equal(o.reshape(-1), want)
    assert lse.reshape(-1)[0] == 0.0


def rand_bits_dtype(shape, seed, dtype):
    rng = np.random.default_rng(seed)
    return fa_inputs.f32_to_bits(rng.standard_normal(shape).astype(np.float32), dtype)


# --------------------------------------------------------------------------- grouped-query attention
@pytest.mark.parametrize("H,Hkv", [(6, 2), (4, 1), (8, 8)])
@pytest.mark.parametrize("causal", [False, True])
def test_gqa_equals_mha_with_each_kv_head_shared_by_its_group(H, Hkv, causal):
    """"Flash Attention 4", section "GQA 支持": the G = H / H_kv consecutive query
    heads kv*G .. kv*G+G-1 all read K/V head kv. Giving every query head its own
    copy of that K/V head must change nothing, bit for bit."""
    B, N, d = 2, 37, 16
    q = rand_bits_dtype((B, N, H, d), 50, "bf16")
    k = rand_bits_dtype((B, N, Hkv, d), 51, "bf16")
    v = rand_bits_dtype((B, N, Hkv, d), 52, "bf16")
    G = H // Hkv
    o, lse = oracle.attention(q, k, v, 0.3, causal)
    o2, lse2 = oracle.attention(q, np.repeat(k, G, axis=2), np.repeat(v, G, axis=2), 0.3, causal)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)
    rows = np.array([[0, 0, 0], [1, H - 1, N - 1], [0, H // 2, 20]], np.int64)
    orow, lrow = oracle.attention_rows(q, k, v, rows, 0.3, causal)
    for r, (b, h, i) in enumerate(rows):
        np.testing.assert_array_equal(orow[r], o[b, i, h])
        assert lrow[r] == lse[b, h, i]


def test_gqa_varlen_equals_mha_varlen():
    lengths = [9, 0, 70, 1]
    H, Hkv, d = 6, 3, 8
    _, cu, q, k, v = fa_inputs.make_varlen_from_lengths(lengths, H, d, seed=53, Hkv=Hkv)
    assert k.shape == (sum(lengths), Hkv, d)
    for causal in (False, True):
        o, lse = oracle.attention_varlen(q, k, v, cu, 0.25, causal)
        o2, lse2 = oracle.attention_varlen(q, np.repeat(k, 2, axis=1), np.repeat(v, 2, axis=1), cu, 0.25, causal)
        np.testing.assert_array_equal(o, o2)
        np.testing.assert_array_equal(lse, lse2)
        rows = np.array([[0, 0], [5, 8], [4, 9], [1, 79]], np.int64)
        orow, lrow = oracle.attention_rows_varlen(q, k, v, cu, rows, 0.25, causal)
        for r, (h, t) in enumerate(rows):
            np.testing.assert_array_equal(orow[r], o[t, h])
            assert lrow[r] == lse[h, t]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("causal", [False, True])
def test_gqa_matches_float64_sdpa(dtype, causal):
    """The pages' own check ("编译与验证"): PyTorch SDPA with enable_gqa, here in float64."""
    torch = pytest.importorskip("torch")
    B, N, H, Hkv, d = 1, 96, 8, 2, 64
    q = rand_bits_dtype((B, N, H, d), 60, dtype)
    k = rand_bits_dtype((B, N, Hkv, d), 61, dtype)
    v = rand_bits_dtype((B, N, Hkv, d), 62, dtype)
    scale = 1.0 / math.sqrt(d)
    o, lse = oracle.attention(q, k, v, scale, causal, dtype=dtype)
    t = lambda b: torch.from_numpy(fa_inputs.bits_to_f32(b, dtype).astype(np.float64)).permute(0, 2, 1, 3)  # noqa: E731
    ref = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), scale=scale, is_causal=causal,
                                                           enable_gqa=True)
    np.testing.assert_allclose(o, ref.permute(0, 2, 1, 3).numpy(), atol=1e-12, rtol=0)
    s = torch.einsum("bhid,bhjd->bhij", t(q), t(k).repeat_interleave(H // Hkv, dim=1)) * scale
    if causal:
        s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), atol=1e-12, rtol=0)


def test_gqa_and_dtype_arguments_are_checked():
    q = np.zeros((1, 4, 6, 8), np.uint16)
    k = np.zeros((1, 4, 4, 8), np.uint16)
    with pytest.raises(ValueError):
        oracle.attention(q, k, k, 0.5, False)          # 6 query heads over 4 K/V heads
    with pytest.raises(ValueError):
        oracle.attention(q, q, q, 0.5, False, dtype="f32")


# --------------------------------------------------------------------------- merging partial results
def test_lse_combine_reproduces_the_two_round_example():
    """The two rounds of "FlashAttention：一次前向计算" (figs. 5-10) taken as two
    separate parts: round 1 = keys {0,1} (numerator fig. 6, denominators 3/2, max 1),
    round 2 alone = keys {2,3} (weights fig. 7 against max 2, which is also each
    row's own max over those keys; numerator fig. 8). Normalising each part and
    merging through LSE must give the printed final output (fig. 10) and
    L = ln 8, ln 9."""
    g = fixtures.load("p3_two_round_example.txt")
    l1 = as_float([g["l1"]])[0]
    m1, m2 = as_float([g["m1"]])[0], as_float([g["m2"]])[0]
    l2_alone = as_float(g["P2"]).sum(axis=1)                  # 5/4, 3/2 (printed after fig. 7)
    o_parts = np.stack([as_float(g["O1"]) / l1[:, None], as_float(g["PV2"]) / l2_alone[:, None]])
    lse_parts = np.stack([LN2 * m1 + np.log(l1), LN2 * m2 + np.log(l2_alone)])
    o, lse = oracle.lse_combine(o_parts, lse_parts)
    np.testing.assert_allclose(o, as_float(g["O"]), rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, [math.log(float(x)) for x in g["LSE_ln"]], rtol=0, atol=1e-14)
    # the oracle on each round's keys alone gives the same parts
    q, k, v = (bits(as_float(g[n])) for n in ("Q", "K", "V"))
    for part, (a, b) in enumerate(((0, 2), (2, 4))):
        op, lp = oracle.attention(one_head(q), one_head(k[a:b]), one_head(v[a:b]), scale=LN2, causal=False)
        np.testing.assert_allclose(op[0, :, 0], o_parts[part], rtol=0, atol=1e-14)
        np.testing.assert_allclose(lp[0, 0], lse_parts[part], rtol=0, atol=1e-14)


@pytest.mark.parametrize("n_parts", [1, 2, 5])
def test_lse_combine_of_key_shards_equals_attention_over_all_keys(n_parts):
    B, N, Nkv, H, d = 1, 40, 203, 2, 32
    rng = np.random.default_rng(70 + n_parts)
    q, k, v = (fa_inputs.f32_to_bf16_bits(rng.standard_normal(s).astype(np.float32))
               for s in ((B, N, H, d), (B, Nkv, H, d), (B, Nkv, H, d)))
    o_all, l_all = oracle.attention(q, k, v, 0.2, False)
    cuts = np.linspace(0, Nkv, n_parts + 1).astype(int)
    parts = [oracle.attention(q, k[:, a:b], v[:, a:b], 0.2, False) for a, b in zip(cuts, cuts[1:])]
    o_parts = np.stack([p[0][0].transpose(1, 0, 2).reshape(H * N, d) for p in parts])   # rows (h, i)
    lse_parts = np.stack([p[1][0].reshape(H * N) for p in parts])
    o, lse = oracle.lse_combine(o_parts, lse_parts)
    np.testing.assert_allclose(o, o_all[0].transpose(1, 0, 2).reshape(H * N, d), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, l_all[0].reshape(H * N), rtol=0, atol=1e-13)


def test_lse_combine_skips_parts_without_keys():
    o_parts = np.array([[[1.0, 2.0], [np.nan, np.inf]], [[3.0, -1.0], [np.nan, 5.0]]])   # [P=2, R=2, d=2]
    lse_parts = np.array([[0.5, -np.inf], [-np.inf, -np.inf]])
    o, lse = oracle.lse_combine(o_parts, lse_parts)
    np.testing.assert_array_equal(o, [[1.0, 2.0], [0.0, 0.0]])     # row 0: part 0 only; row 1: nothing
    np.testing.assert_array_equal(lse, [0.5, -np.inf])
    with pytest.raises(ValueError):
        oracle.lse_combine(o_parts, np.array([[np.nan, 0.0], [0.0, 0.0]]))
