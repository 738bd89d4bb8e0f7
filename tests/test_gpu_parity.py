"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances (max-abs, for bf16 inputs, independent of tau): O <= 2e-2, LSE <= 1e-3.
Small and ragged shapes are compared element by element; the full-size
workloads are compared on sampled rows that the oracle computes one by one.
"""
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
    fa.set_option("tau", 8.0)
    fa.set_option("persistent", -1)
    fa.set_option("exp2_emulation", 0)


@pytest.fixture(params=["two_tile", "auto"], autouse=True)
def task_shape(request):
    """Every test twice: with two-tile tasks forced, and with the library's choice
    (small shapes then run as solo tasks)."""
    fa.set_option("solo_tiles", 0 if request.param == "two_tile" else -1)
    yield request.param
    fa.set_option("solo_tiles", -1)


def dev(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def host(t):
    import torch
    if t.dtype == torch.bfloat16:
        return fa_inputs.bf16_bits_to_f32(t.view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)
    return t.cpu().numpy().astype(np.float64)


def run_fixed(q, k, v, causal, scale=None, lse=True):
    import torch
    out = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    B, N, H, d = q.shape
    l = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda") if lse else None
    fa.fa_fwd(dev(q), dev(k), dev(v), scale=scale, causal=causal, out=out, lse=l, return_lse=lse)
    st, word = fa.last_device_status()
    assert st == fa.FA_OK, hex(word)
    return host(out), (host(l) if lse else None)


def check(o, lse, o_ref, lse_ref, what=""):
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    err_o = np.abs(o - o_ref).max()
    assert err_o <= TOL_O, f"{what}: max |O - oracle| = {err_o}"
    if lse is not None:
        fin = np.isfinite(lse_ref)
        assert np.array_equal(np.isfinite(lse), fin), f"{what}: LSE finiteness differs"
        err_l = np.abs(lse[fin] - lse_ref[fin]).max() if fin.any() else 0.0
        assert err_l <= TOL_LSE, f"{what}: max |LSE - oracle| = {err_l}"
    return err_o


# --------------------------------------------------------------------------- building blocks
@pytest.mark.parametrize("d", [64, 128])
def test_mma_tile_plumbing(d):
    rng = np.random.default_rng(d)
    q, k, v, p = (fa_inputs.f32_to_bf16_bits(rng.standard_normal(s).astype(np.float32))
                  for s in ((128, d), (128, d), (128, d), (128, 128)))
    s_gpu, o_gpu = fa.selftest_mma_tile(dev(q), dev(k), dev(v), dev(p))
    f = lambda b: fa_inputs.bf16_bits_to_f32(b).astype(np.float64)  # noqa: E731
    s_ref = f(q) @ f(k).T
    o_ref = f(p) @ f(v)
    assert np.abs(host(s_gpu) - s_ref).max() < 1e-3 * max(1.0, np.abs(s_ref).max())
    assert np.abs(host(o_gpu) - o_ref).max() < 1e-3 * max(1.0, np.abs(o_ref).max())


def test_exp2_paths():
    import torch
    x = torch.linspace(-40.0, 8.0, 1 << 20, device="cuda", dtype=torch.float32)
    ref = np.exp2(x.cpu().numpy().astype(np.float64))
    hw = host(fa.selftest_exp2(x, False))
    poly = host(fa.selftest_exp2(x, True))
    assert np.abs(hw / ref - 1).max() < 1e-6
    assert np.abs(poly / ref - 1).max() < 2e-4
    poly2 = host(fa.selftest_exp2(x, 2))
    assert np.array_equal(poly2, poly)
    # very negative and -inf inputs: hardware path gives 0, polynomial a tiny non-negative value
    y = host(fa.selftest_exp2(torch.tensor([-float("inf"), -200.0, -127.0], device="cuda"), False))
    assert y[0] == 0.0 and y[1] == 0.0
    y = host(fa.selftest_exp2(torch.tensor([-float("inf"), -200.0], device="cuda"), True))
    assert (y >= 0).all() and (y < 2.0 ** -124).all()


def test_bounded_wait_times_out_and_context_survives():
    assert fa.selftest_wait_timeout(20_000_000) == fa.FA_ERR_TIMEOUT
    q, k, v = fa_inputs.make_qkv(1, 128, 1, 64, seed=3)
    o, lse = run_fixed(q, k, v, causal=True)
    o_ref, l_ref = oracle.attention(q, k, v, 1 / 8, True)
    check(o, lse, o_ref, l_ref, "after timeout")


# --------------------------------------------------------------------------- small and ragged shapes
SHAPES = [(1, 1, 1, 64), (1, 1, 7, 128), (1, 2, 128, 64), (2, 1, 129, 128), (1, 3, 255, 64),
          (1, 1, 256, 128), (2, 2, 300, 128), (1, 1, 640, 64), (1, 2, 1000, 128), (3, 1, 513, 64)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%dH%dN%dd%d" % s)
def test_fixed_length_elementwise(shape, causal):
    B, H, N, d = shape
    q, k, v = fa_inputs.make_qkv(B, N, H, d, seed=1000 + N + d)
    o, lse = run_fixed(q, k, v, causal)
    o_ref, l_ref = oracle.attention(q, k, v, 1 / math.sqrt(d), causal)
    check(o, lse, o_ref, l_ref, f"{shape} causal={causal}")


@pytest.mark.parametrize("tau", [0.0, 8.0, 16.0])
@pytest.mark.parametrize("emu", [0, 4, 8])
def test_spiky_inputs_independent_of_tau_and_exp_path(tau, emu):
    """Spiky scores (the delayed rescale fires): same result for any tau whose
    bound 2^tau on the unnormalised weights stays inside fp32."""
    fa.set_option("tau", tau)
    fa.set_option("exp2_emulation", emu)
    try:
        q, k, v = fa_inputs.make_qkv(1, 1100, 2, 128, seed=20264, spiky=True)
        o, lse = run_fixed(q, k, v, True)
    finally:
        fa.set_option("tau", 8.0)
        fa.set_option("exp2_emulation", 0)
    o_ref, l_ref = oracle.attention(q, k, v, 1 / math.sqrt(128), True)
    check(o, lse, o_ref, l_ref, f"tau={tau} emu={emu}")


@pytest.mark.parametrize("tau", [0.0, 8.0, math.inf])
@pytest.mark.parametrize("causal", [False, True])
def test_unit_normal_inputs_independent_of_tau(tau, causal):
    """tau = inf never rescales after the first block; with N(0,1) inputs the
    weights stay far inside fp32, so the result must not change."""
    fa.set_option("tau", tau)
    try:
        q, k, v = fa_inputs.make_qkv(1, 1500, 2, 128, seed=31)
        o, lse = run_fixed(q, k, v, causal)
    finally:
        fa.set_option("tau", 8.0)
    o_ref, l_ref = oracle.attention(q, k, v, 1 / math.sqrt(128), causal)
    check(o, lse, o_ref, l_ref, f"tau={tau}")


@pytest.mark.parametrize("causal", [False, True])
def test_scheduling_modes_agree_bitwise(causal):
    """One task per CTA, static stride and work stealing give identical bits."""
    q, k, v = fa_inputs.make_qkv(2, 700, 3, 128, seed=77)
    outs = []
    for mode in (0, 1, 2):
        fa.set_option("persistent", mode)
        try:
            outs.append(run_fixed(q, k, v, causal))
        finally:
            fa.set_option("persistent", -1)
    for o, l in outs[1:]:
        assert np.array_equal(outs[0][0], o)
        assert np.array_equal(outs[0][1], l)


def test_deterministic_and_lse_optional():
    q, k, v = fa_inputs.make_qkv(1, 333, 2, 64, seed=5)
    a = run_fixed(q, k, v, True)
    b = run_fixed(q, k, v, True)
    c = run_fixed(q, k, v, True, lse=False)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and np.array_equal(a[0], c[0])


def test_scale_argument_is_used():
    q, k, v = fa_inputs.make_qkv(1, 200, 1, 64, seed=6)
    o, lse = run_fixed(q, k, v, False, scale=0.5)
    o_ref, l_ref = oracle.attention(q, k, v, 0.5, False)
    check(o, lse, o_ref, l_ref, "scale=0.5")


def test_output_rows_only_inside_the_tensor():
    """A canary after O and LSE stays untouched (no store past the last row)."""
    import torch
    B, N, H, d = 1, 130, 2, 128
    q, k, v = fa_inputs.make_qkv(B, N, H, d, seed=8)
    big = torch.full((B * N * H * d + 4096,), 7.0, dtype=torch.bfloat16, device="cuda")
    lbig = torch.full((B * H * N + 1024,), 7.0, dtype=torch.float32, device="cuda")
    out = big[: B * N * H * d].view(B, N, H, d)
    l = lbig[: B * H * N].view(B, H, N)
    fa.fa_fwd(dev(q), dev(k), dev(v), causal=True, out=out, lse=l)
    torch.cuda.synchronize()
    assert (big[B * N * H * d:] == 7.0).all() and (lbig[B * H * N:] == 7.0).all()
    o_ref, l_ref = oracle.attention(q, k, v, 1 / math.sqrt(d), True)
    check(host(out), host(l), o_ref, l_ref, "canary")


# --------------------------------------------------------------------------- varlen
def run_varlen(lengths, H, d, causal, seed):
    import torch
    _, cu, q, k, v = fa_inputs.make_varlen_from_lengths(lengths, H, d, seed)
    T = int(cu[-1])
    out = torch.full((T, H, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    l = torch.full((H, T), float("nan"), dtype=torch.float32, device="cuda")
    cu_d = torch.from_numpy(cu).cuda()
    fa.fa_fwd_varlen(dev(q), dev(k), dev(v), cu_d, max(max(lengths), 1), causal=causal, out=out, lse=l)
    st, word = fa.last_device_status()
    assert st == fa.FA_OK, hex(word)
    return (q, k, v, cu), host(out), host(l)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("lengths", [[1], [7, 0, 129], [128, 256, 1], [300, 5, 0, 700, 64], [0, 0, 3]],
                         ids=str)
def test_varlen_elementwise(lengths, causal):
    (q, k, v, cu), o, lse = run_varlen(lengths, 3, 128, causal, seed=sum(lengths))
    o_ref, l_ref = oracle.attention_varlen(q, k, v, cu, 1 / math.sqrt(128), causal)
    check(o, lse, o_ref, l_ref, f"varlen {lengths}")


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_short_last_blocks(causal):
    """Sequences whose last 256-row block holds 128 rows or fewer (a task of one Q tile
    at the sequence's end): remainders of 1, 44, 128 and 129 rows, sequences of one
    tile, and one long sequence with a full last block."""
    lengths = [257, 300, 640, 385, 129, 1, 128, 384, 2000]
    (q, k, v, cu), o, lse = run_varlen(lengths, 2, 128, causal, seed=77)
    o_ref, l_ref = oracle.attention_varlen(q, k, v, cu, 1 / math.sqrt(128), causal)
    check(o, lse, o_ref, l_ref, f"varlen short last blocks causal={causal}")


@pytest.mark.parametrize("N,Nk,H,Hkv,splits", [(300, 300, 2, 2, 1), (1100, 1100, 4, 1, 1), (4100, 4100, 2, 2, 1),
                                               (385, 700, 8, 2, 1), (1100, 1100, 2, 2, 3)], ids=str)
def test_fixed_length_short_last_blocks(N, Nk, H, Hkv, splits):
    """Causal fixed-length problems whose last 256-row block holds 128 packed rows or
    fewer (a task of one Q tile), with grouped heads, N_q != N_kv and key splits: every
    element against the oracle."""
    import torch
    q, k, v = fa_inputs.make_qkv(1, N, H, 128, seed=N + H, Hkv=Hkv, Nkv=Nk)
    out = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    l = torch.full((1, H, N), float("nan"), dtype=torch.float32, device="cuda")
    fa.fa_fwd(dev(q), dev(k), dev(v), causal=True, out=out, lse=l, num_splits=splits)
    st, word = fa.last_device_status()
    assert st == fa.FA_OK, hex(word)
    o_ref, l_ref = oracle.attention(q, k, v, 1 / math.sqrt(128), True)
    check(host(out), host(l), o_ref, l_ref, f"N={N} N_kv={Nk} H={H}/{Hkv} splits={splits}")


def test_varlen_d64():
    (q, k, v, cu), o, lse = run_varlen([200, 77, 513], 2, 64, True, seed=9)
    o_ref, l_ref = oracle.attention_varlen(q, k, v, cu, 1 / 8, True)
    check(o, lse, o_ref, l_ref, "varlen d64")


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_schedule_is_complete_and_longest_first(causal):
    import torch
    lengths = [300, 5, 0, 700, 64, 1, 2000]
    H = 3
    cu = np.zeros(len(lengths) + 1, np.int32)
    cu[1:] = np.cumsum(lengths)
    tasks, n = fa.varlen_schedule(torch.from_numpy(cu).cuda(), H, causal, capacity=4096)
    t = tasks.cpu().numpy()
    want = set()
    for s, L in enumerate(lengths):
        for m in range((L + 255) // 256):
            for h in range(H):
                want.add((s, h, m))
    assert n == len(want) and {tuple(x[:3]) for x in t} == want
    cost = t[:, 3]
    assert (np.diff(cost) <= 0).all()
    for s, h, m, c in t:
        kmax = min(m * 256 + 256, lengths[s]) if causal else lengths[s]
        assert c == (kmax + 127) // 128


# --------------------------------------------------------------------------- the five workloads
def sample_rows(B, H, N, n_rand, seed):
    rng = np.random.default_rng(seed)
    fixed = sorted({0, 1, 127, 128, 129, 255, 256, N // 2, N - 129, N - 128, N - 2, N - 1} & set(range(N)))
    rows = []
    for b in range(B):
        for h in range(H):
            pick = set(fixed) | set(rng.integers(0, N, n_rand).tolist())
            rows += [(b, h, i) for i in sorted(pick)]
    return np.array(rows, np.int64)


@pytest.mark.parametrize("name", ["c1_b1h1n256d64", "c2_b2h8n1024d128"])
def test_small_workloads_elementwise(name):
    w = fa_inputs.WORKLOADS[name]
    x = fa_inputs.make_workload(w)
    o, lse = run_fixed(x["q"], x["k"], x["v"], w.causal, scale=w.scale)
    o_ref, l_ref = oracle.attention(x["q"], x["k"], x["v"], w.scale, w.causal)
    check(o, lse, o_ref, l_ref, name)


@pytest.mark.parametrize("name", ["c3_b4h16n4096d128_causal", "c4_b1h32n16384d128_causal_spiky"])
def test_large_workloads_sampled_rows(name):
    w = fa_inputs.WORKLOADS[name]
    x = fa_inputs.make_workload(w)
    o, lse = run_fixed(x["q"], x["k"], x["v"], w.causal, scale=w.scale)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    rows = sample_rows(w.B, w.H, w.N, 16, w.seed)
    o_ref, l_ref = oracle.attention_rows(x["q"], x["k"], x["v"], rows, w.scale, w.causal)
    b, h, i = rows.T
    check(o[b, i, h], lse[b, h, i], o_ref, l_ref, name)


def test_varlen_workload_sampled_rows():
    import torch
    w = fa_inputs.WORKLOADS["c5_varlen8_h16d128_causal"]
    x = fa_inputs.make_workload(w)
    cu = x["cu_seqlens"]
    T = int(cu[-1])
    o, l = fa.fa_fwd_varlen(dev(x["q"]), dev(x["k"]), dev(x["v"]), torch.from_numpy(cu).cuda(),
                            int(x["lengths"].max()), scale=w.scale, causal=True)
    assert fa.last_device_status()[0] == fa.FA_OK
    o, l = host(o), host(l)
    assert np.isfinite(o).all() and np.isfinite(l).all()
    rng = np.random.default_rng(w.seed)
    rows = []
    for s in range(len(x["lengths"])):
        a, b = int(cu[s]), int(cu[s + 1])
        toks = {a, a + 1, a + 127, a + 128, a + 255, a + 256, b - 1, b - 2} | set(rng.integers(a, b, 8).tolist())
        rows += [(h, t) for h in range(w.H) for t in sorted(toks) if a <= t < b]
    rows = np.array(rows, np.int64)
    o_ref, l_ref = oracle.attention_rows_varlen(x["q"], x["k"], x["v"], cu, rows, w.scale, True)
    h, t = rows.T
    check(o[t, h], l[h, t], o_ref, l_ref, "c5 varlen")
    assert T == o.shape[0]
