"""GPU parity for grouped-query attention and fp16 inputs ("Flash Attention 4",
sections "GQA 支持" and "编译与验证"): the CUDA path through the C ABI against
the fp64 oracle.

The kernel packs the G = H / H_kv query heads that share a K/V head into the
rows of each 128-row Q tile (128 / G positions x G heads). The cases below cover
every group size class (G = 1, 2, 4, 8, 32, 128: one position per tile), ragged
sequence ends inside a packed tile, both masks, both head dims and both element
types. Tolerances as for the bf16 multi-head path: O <= 2e-2, LSE <= 1e-3 max-abs.
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


@pytest.fixture(params=["two_tile", "auto"], autouse=True)
def task_shape(request):
    """Every test twice: with two-tile tasks forced, and with the library's choice
    (small shapes then run as solo tasks)."""
    fa.set_option("solo_tiles", 0 if request.param == "two_tile" else -1)
    yield request.param
    fa.set_option("solo_tiles", -1)


def tdtype(dtype):
    import torch
    return torch.float16 if dtype == "f16" else torch.bfloat16


def dev(bits, dtype="bf16"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(tdtype(dtype)).cuda()


def host(t):
    import torch
    if t.dtype in (torch.bfloat16, torch.float16):
        dtype = "f16" if t.dtype == torch.float16 else "bf16"
        return fa_inputs.bits_to_f32(t.view(torch.int16).cpu().numpy().view(np.uint16), dtype).astype(np.float64)
    return t.cpu().numpy().astype(np.float64)


def check(o, lse, o_ref, lse_ref, what=""):
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    err_o = np.abs(o - o_ref).max()
    assert err_o <= TOL_O, f"{what}: max |O - oracle| = {err_o}"
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse), fin), f"{what}: LSE finiteness differs"
    err_l = np.abs(lse[fin] - lse_ref[fin]).max() if fin.any() else 0.0
    assert err_l <= TOL_LSE, f"{what}: max |LSE - oracle| = {err_l}"


def run_fixed(q, k, v, causal, dtype, scale=None):
    import torch
    B, N, H, d = q.shape
    out = torch.full(q.shape, float("nan"), dtype=tdtype(dtype), device="cuda")
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
    fa.fa_fwd(dev(q, dtype), dev(k, dtype), dev(v, dtype), scale=scale, causal=causal, out=out, lse=lse)
    st, word = fa.last_device_status()
    assert st == fa.FA_OK, hex(word)
    return host(out), host(lse)


# --------------------------------------------------------------------------- building block
@pytest.mark.parametrize("d", [64, 128])
def test_mma_tile_plumbing_fp16(d):
    rng = np.random.default_rng(100 + d)
    q, k, v, p = (fa_inputs.f32_to_f16_bits(rng.standard_normal(s).astype(np.float32))
                  for s in ((128, d), (128, d), (128, d), (128, 128)))
    s_gpu, o_gpu = fa.selftest_mma_tile(dev(q, "f16"), dev(k, "f16"), dev(v, "f16"), dev(p, "f16"))
    f = lambda b: fa_inputs.f16_bits_to_f32(b).astype(np.float64)  # noqa: E731
    s_ref = f(q) @ f(k).T
    o_ref = f(p) @ f(v)
    assert np.abs(host(s_gpu) - s_ref).max() < 1e-4 * max(1.0, np.abs(s_ref).max())
    assert np.abs(host(o_gpu) - o_ref).max() < 1e-4 * max(1.0, np.abs(o_ref).max())


# --------------------------------------------------------------------------- fixed length
GQA_SHAPES = [  # (B, H, H_kv, N, d)
    (1, 4, 1, 300, 128),     # G = 4 (multi-query)
    (2, 8, 2, 129, 64),      # G = 4, ragged tail inside a packed tile
    (1, 16, 2, 1000, 128),   # G = 8
    (1, 6, 3, 513, 128),     # G = 2
    (1, 32, 1, 77, 64),      # G = 32
    (1, 128, 1, 40, 64),     # G = 128: one sequence position per tile
    (1, 4, 4, 333, 128),     # G = 1
]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", GQA_SHAPES, ids=lambda s: "B%dH%dKV%dN%dd%d" % s)
def test_gqa_fixed_length_elementwise(shape, causal, dtype):
    B, H, Hkv, N, d = shape
    q, k, v = fa_inputs.make_qkv(B, N, H, d, seed=2000 + N + H, Hkv=Hkv, dtype=dtype)
    o, lse = run_fixed(q, k, v, causal, dtype)
    o_ref, l_ref = oracle.attention(q, k, v, 1 / math.sqrt(d), causal, dtype=dtype)
    check(o, lse, o_ref, l_ref, f"{shape} causal={causal} {dtype}")


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_scheduling_modes_agree_bitwise(causal):
    q, k, v = fa_inputs.make_qkv(2, 700, 8, 128, seed=78, Hkv=2)
    outs = []
    for mode in (0, 1, 2):
        fa.set_option("persistent", mode)
        try:
            outs.append(run_fixed(q, k, v, causal, "bf16"))
        finally:
            fa.set_option("persistent", -1)
    for o, l in outs[1:]:
        assert np.array_equal(outs[0][0], o) and np.array_equal(outs[0][1], l)


@pytest.mark.parametrize("tau", [0.0, 8.0, 40.0])
def test_fp16_spiky_inputs_with_any_tau(tau):
    """fp16 weights must stay finite: the library caps tau at 15 for fp16, so even
    tau = 40 (weights up to 2^40 without the cap) gives the oracle's result."""
    fa.set_option("tau", tau)
    try:
        q, k, v = fa_inputs.make_qkv(1, 1100, 4, 128, seed=20264, spiky=True, Hkv=2, dtype="f16")
        o, lse = run_fixed(q, k, v, True, "f16")
    finally:
        fa.set_option("tau", 8.0)
    o_ref, l_ref = oracle.attention(q, k, v, 1 / math.sqrt(128), True, dtype="f16")
    check(o, lse, o_ref, l_ref, f"fp16 spiky tau={tau}")


def test_gqa_output_rows_only_inside_the_tensor():
    import torch
    B, N, H, Hkv, d = 1, 67, 8, 2, 128
    q, k, v = fa_inputs.make_qkv(B, N, H, d, seed=81, Hkv=Hkv)
    big = torch.full((B * N * H * d + 4096,), 7.0, dtype=torch.bfloat16, device="cuda")
    lbig = torch.full((B * H * N + 1024,), 7.0, dtype=torch.float32, device="cuda")
    out = big[: B * N * H * d].view(B, N, H, d)
    lse = lbig[: B * H * N].view(B, H, N)
    fa.fa_fwd(dev(q), dev(k), dev(v), causal=True, out=out, lse=lse)
    torch.cuda.synchronize()
    assert (big[B * N * H * d:] == 7.0).all() and (lbig[B * H * N:] == 7.0).all()
    o_ref, l_ref = oracle.attention(q, k, v, 1 / math.sqrt(d), True)
    check(host(out), host(lse), o_ref, l_ref, "gqa canary")


# --------------------------------------------------------------------------- varlen
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("lengths,H,Hkv", [([7, 0, 129, 300], 8, 2), ([1, 64, 33], 16, 1), ([500, 260], 4, 2)],
                         ids=str)
def test_gqa_varlen_elementwise(lengths, H, Hkv, causal, dtype):
    import torch
    _, cu, q, k, v = fa_inputs.make_varlen_from_lengths(lengths, H, 128, seed=sum(lengths) + H, Hkv=Hkv,
                                                        dtype=dtype)
    T = int(cu[-1])
    out = torch.full((T, H, 128), float("nan"), dtype=tdtype(dtype), device="cuda")
    lse = torch.full((H, T), float("nan"), dtype=torch.float32, device="cuda")
    fa.fa_fwd_varlen(dev(q, dtype), dev(k, dtype), dev(v, dtype), torch.from_numpy(cu).cuda(), max(lengths),
                     causal=causal, out=out, lse=lse)
    st, word = fa.last_device_status()
    assert st == fa.FA_OK, hex(word)
    o_ref, l_ref = oracle.attention_varlen(q, k, v, cu, 1 / math.sqrt(128), causal, dtype=dtype)
    check(host(out), host(lse), o_ref, l_ref, f"varlen gqa {lengths} {dtype}")


@pytest.mark.parametrize("group", [2, 4, 128])
def test_gqa_varlen_schedule_covers_packed_rows(group):
    import torch
    lengths = [300, 5, 0, 700, 64, 1]
    Hkv = 3
    cu = np.zeros(len(lengths) + 1, np.int32)
    cu[1:] = np.cumsum(lengths)
    tasks, n = fa.varlen_schedule(torch.from_numpy(cu).cuda(), Hkv, True, capacity=8192, group=group)
    t = tasks.cpu().numpy()
    want = {(s, h, m) for s, L in enumerate(lengths) for m in range((L * group + 255) // 256) for h in range(Hkv)}
    assert n == len(want) and {tuple(x[:3]) for x in t} == want
    assert (np.diff(t[:, 3]) <= 0).all()
    for s, h, m, c in t:
        last_pos = (m * 256 + 255) // group          # the task's last packed row's position
        assert c == (min(last_pos + 1, lengths[s]) + 127) // 128


# --------------------------------------------------------------------------- the GQA workloads
def test_gqa_fp16_workload_elementwise():
    w = fa_inputs.WORKLOADS["g1_gqa_b1h32kv8n1024d128_f16"]
    x = fa_inputs.make_workload(w)
    o, lse = run_fixed(x["q"], x["k"], x["v"], w.causal, w.dtype, scale=w.scale)
    o_ref, l_ref = oracle.attention(x["q"], x["k"], x["v"], w.scale, w.causal, dtype=w.dtype)
    check(o, lse, o_ref, l_ref, w.name)


def test_gqa_causal_workload_sampled_rows():
    w = fa_inputs.WORKLOADS["g2_gqa_b4h32kv8n4096d128_causal"]
    x = fa_inputs.make_workload(w)
    o, lse = run_fixed(x["q"], x["k"], x["v"], w.causal, w.dtype, scale=w.scale)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    rng = np.random.default_rng(w.seed)
    fixed = [0, 1, 31, 32, 63, 64, 127, 128, 2048, w.N - 33, w.N - 32, w.N - 1]
    rows = np.array([(b, h, i) for b in range(w.B) for h in range(w.H)
                     for i in sorted(set(fixed) | set(rng.integers(0, w.N, 6).tolist()))], np.int64)
    o_ref, l_ref = oracle.attention_rows(x["q"], x["k"], x["v"], rows, w.scale, w.causal, dtype=w.dtype)
    b, h, i = rows.T
    check(o[b, i, h], lse[b, h, i], o_ref, l_ref, w.name)


def test_gqa_fp16_varlen_workload_sampled_rows():
    import torch
    w = fa_inputs.WORKLOADS["g3_gqa_varlen8_h32kv4d128_causal_f16"]
    x = fa_inputs.make_workload(w)
    cu = x["cu_seqlens"]
    o, lse = fa.fa_fwd_varlen(dev(x["q"], "f16"), dev(x["k"], "f16"), dev(x["v"], "f16"),
                              torch.from_numpy(cu).cuda(), int(x["lengths"].max()), scale=w.scale, causal=True)
    assert fa.last_device_status()[0] == fa.FA_OK
    o, lse = host(o), host(lse)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    rng = np.random.default_rng(w.seed)
    rows = []
    for s in range(len(x["lengths"])):
        a, b = int(cu[s]), int(cu[s + 1])
        toks = {a, a + 1, a + 15, a + 16, a + 31, a + 32, b - 1, b - 2} | set(rng.integers(a, b, 4).tolist())
        rows += [(h, t) for h in range(w.H) for t in sorted(toks) if a <= t < b]
    rows = np.array(rows, np.int64)
    o_ref, l_ref = oracle.attention_rows_varlen(x["q"], x["k"], x["v"], cu, rows, w.scale, True, dtype="f16")
    h, t = rows.T
    check(o[t, h], lse[h, t], o_ref, l_ref, w.name)
