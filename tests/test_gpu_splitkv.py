"""GPU parity for N_q != N_kv, key splits merged through the LSE, and the
standalone merge (fa_lse_combine), against the fp64 oracle.

* N_q != N_kv follows the bottom-right causal alignment of "Flash Attention 4",
  section "Causal Mask" (query i sees keys j <= i + N_kv - N_q); rows that see
  no key (N_q > N_kv) must come back as O = 0, LSE = -inf.
* With num_splits > 1 every task's keys are cut into ranges computed as
  separate tasks and merged by LSE ("FlashAttention：一次前向计算", two-round
  example): the result must match the oracle over all keys.
Tolerances as everywhere: O <= 2e-2, LSE <= 1e-3 max-abs.
"""
import math

import numpy as np
import pytest

import attention_forward_tma_gb300 as fa
import fa_inputs
import oracle
from tests.golden import fixtures

pytestmark = pytest.mark.gpu

TOL_O = 2e-2
TOL_LSE = 1e-3


@pytest.fixture(scope="module", autouse=True)
def cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.library()
    yield torch
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
    assert (lse[~fin] == -np.inf).all(), f"{what}: rows without keys must have LSE = -inf"
    err_l = np.abs(lse[fin] - lse_ref[fin]).max() if fin.any() else 0.0
    assert err_l <= TOL_LSE, f"{what}: max |LSE - oracle| = {err_l}"


def run_kv(q, k, v, causal, dtype="bf16", splits=1):
    import torch
    B, N, H, d = q.shape
    out = torch.full(q.shape, float("nan"), dtype=tdtype(dtype), device="cuda")
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
    fa.fa_fwd(dev(q, dtype), dev(k, dtype), dev(v, dtype), causal=causal, out=out, lse=lse, num_splits=splits)
    st, word = fa.last_device_status()
    assert st == fa.FA_OK, hex(word)
    return host(out), host(lse)


# --------------------------------------------------------------------------- N_q != N_kv
KV_SHAPES = [  # (B, H, H_kv, N_q, N_kv, d)
    (1, 2, 2, 100, 300, 128),    # more keys than queries: rows see 201..300 keys (causal)
    (2, 4, 1, 1, 1000, 64),      # one query row per sequence (decoding), multi-query
    (1, 8, 2, 33, 513, 128),     # ragged both ways, G = 4
    (1, 2, 2, 300, 100, 128),    # more queries than keys: causal rows 0..199 see nothing
    (1, 1, 1, 129, 1, 64),       # a single key
]


@pytest.mark.parametrize("splits", [1, 3])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", KV_SHAPES, ids=lambda s: "B%dH%dKV%dNq%dNk%dd%d" % s)
def test_nq_ne_nkv_elementwise(shape, causal, splits):
    B, H, Hkv, Nq, Nk, d = shape
    q, k, v = fa_inputs.make_qkv(B, Nq, H, d, seed=3000 + Nq + Nk, Nkv=Nk, Hkv=Hkv)
    o, lse = run_kv(q, k, v, causal, splits=splits)
    o_ref, l_ref = oracle.attention(q, k, v, 1 / math.sqrt(d), causal)
    check(o, lse, o_ref, l_ref, f"{shape} causal={causal} splits={splits}")


@pytest.mark.parametrize("splits", [2, 5, 16, 0, 1000])
@pytest.mark.parametrize("causal", [False, True])
def test_key_splits_match_the_oracle(splits, causal):
    """Several ranges per task, including more ranges than some tasks have blocks
    (causal top rows) and a request above the number of key blocks (capped)."""
    q, k, v = fa_inputs.make_qkv(2, 700, 8, 128, seed=91, Hkv=2, dtype="f16")
    o, lse = run_kv(q, k, v, causal, "f16", splits)
    o_ref, l_ref = oracle.attention(q, k, v, 1 / math.sqrt(128), causal, dtype="f16")
    check(o, lse, o_ref, l_ref, f"splits={splits} causal={causal}")


def test_split_and_unsplit_agree_closely():
    q, k, v = fa_inputs.make_qkv(1, 64, 16, 128, seed=92, Nkv=5000, Hkv=4)
    a = run_kv(q, k, v, True, splits=1)
    b = run_kv(q, k, v, True, splits=7)
    assert np.abs(a[0] - b[0]).max() <= 2 * 2.0 ** -8
    assert np.abs(a[1] - b[1]).max() <= 1e-4


def test_release_cached_memory_between_calls():
    """The split partials come from the library's pool, which keeps them between calls;
    fa_release_cached_memory hands them back (device free memory grows by at least the
    partials' size) and the next call allocates afresh with the same result."""
    import torch
    q, k, v = fa_inputs.make_qkv(1, 4096, 32, 128, seed=93, Nkv=8192, Hkv=8)
    qd, kd, vd = dev(q), dev(k), dev(v)
    splits = 8
    partial_bytes = splits * 4096 * 32 * (128 + 1) * 4      # fp32 O and LSE per key range
    a = fa.fa_fwd(qd, kd, vd, causal=True, num_splits=splits)
    torch.cuda.synchronize()
    free_kept = torch.cuda.mem_get_info()[0]
    fa.release_cached_memory()
    free_released = torch.cuda.mem_get_info()[0]
    assert free_released - free_kept >= partial_bytes
    b = fa.fa_fwd(qd, kd, vd, causal=True, num_splits=splits)
    st, word = fa.last_device_status()
    assert st == fa.FA_OK, hex(word)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    fa.release_cached_memory()


def test_spiky_scores_with_splits():
    """Large score gaps across ranges: each range has its own reference, the merge rescales."""
    q, k, v = fa_inputs.make_qkv(1, 200, 4, 128, seed=20264, spiky=True, Nkv=3000)
    o, lse = run_kv(q, k, v, True, splits=6)
    o_ref, l_ref = oracle.attention(q, k, v, 1 / math.sqrt(128), True)
    check(o, lse, o_ref, l_ref, "spiky splits")


# --------------------------------------------------------------------------- varlen with own key lengths
@pytest.mark.parametrize("splits", [1, 3])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("lq,lk", [([1, 1, 1], [700, 1, 129]), ([100, 0, 7, 300], [300, 5, 0, 300]),
                                   ([260, 40], [130, 900])], ids=str)
def test_varlen_kv_elementwise(lq, lk, causal, splits):
    import torch
    H, Hkv, d = 8, 2, 128
    rng = np.random.default_rng(sum(lq) + 7 * sum(lk))
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    mk = lambda n, h: fa_inputs.f32_to_bf16_bits(rng.standard_normal((n, h, d)).astype(np.float32))  # noqa: E731
    q, k, v = mk(int(cu_q[-1]), H), mk(int(cu_k[-1]), Hkv), mk(int(cu_k[-1]), Hkv)
    out = torch.full((int(cu_q[-1]), H, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((H, int(cu_q[-1])), float("nan"), dtype=torch.float32, device="cuda")
    fa.fa_fwd_varlen(dev(q), dev(k), dev(v), torch.from_numpy(cu_q).cuda(), max(lq), causal=causal, out=out,
                     lse=lse, cu_seqlens_k=torch.from_numpy(cu_k).cuda(), max_seqlen_k=max(lk), num_splits=splits)
    st, word = fa.last_device_status()
    assert st == fa.FA_OK, hex(word)
    o_ref = np.zeros((int(cu_q[-1]), H, d))
    l_ref = np.full((H, int(cu_q[-1])), -np.inf)
    for s in range(len(lq)):
        a, b, ka, kb = cu_q[s], cu_q[s + 1], cu_k[s], cu_k[s + 1]
        if b == a or kb == ka:
            continue
        os_, ls_ = oracle.attention(q[None, a:b], k[None, ka:kb], v[None, ka:kb], 1 / math.sqrt(d), causal)
        o_ref[a:b], l_ref[:, a:b] = os_[0], ls_[0]
    check(host(out), host(lse), o_ref, l_ref, f"varlen kv {lq} {lk}")


@pytest.mark.parametrize("splits", [1, 4])
def test_varlen_schedule_with_key_ranges(splits):
    import torch
    lq, lk = [300, 5, 0, 64, 1], [300, 900, 7, 0, 5000]
    cu_q = torch.from_numpy(np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)).cuda()
    cu_k = torch.from_numpy(np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)).cuda()
    tasks, n = fa.varlen_schedule(cu_q, 2, True, capacity=4096, group=4, cu_seqlens_k=cu_k, splits=splits)
    t = tasks.cpu().numpy()
    want = {(s, h | (sp << 16), m) for s, L in enumerate(lq) for m in range((L * 4 + 255) // 256)
            for h in range(2) for sp in range(splits)}
    assert n == len(want) and {tuple(x[:3]) for x in t} == want
    assert (np.diff(t[:, 3]) <= 0).all()
    for s, hs, m, c in t:
        sp = hs >> 16
        off = lk[s] - lq[s]
        kmax = min((m * 256 + 255) // 4 + off + 1, lk[s])
        nb = (kmax + 127) // 128 if kmax > 0 else 0
        per = -(-((lk[s] + 127) // 128) // splits)
        lo, hi = (0, nb) if splits == 1 else (sp * per, max(sp * per, min(sp * per + per, nb)))
        assert c == hi - lo


# --------------------------------------------------------------------------- the merge on its own
def test_lse_combine_matches_oracle():
    import torch
    P, B, N, H, d = 4, 2, 37, 3, 128
    rng = np.random.default_rng(5)
    o_parts = rng.standard_normal((P, B, N, H, d)).astype(np.float32)
    lse_parts = (rng.standard_normal((P, B, H, N)) * 20).astype(np.float32)
    lse_parts[1, 0, 0, :5] = -np.inf               # some parts saw no key
    lse_parts[:, 1, 2, 7] = -np.inf                # a row that saw nothing at all
    o_parts[1, 0, :5, 0] = np.nan                  # never read: its LSE is -inf
    o, lse = fa.lse_combine(torch.from_numpy(o_parts).cuda(), torch.from_numpy(lse_parts).cuda())
    assert fa.last_device_status()[0] == fa.FA_OK
    rows = lambda x: np.moveaxis(x, -1, 2)  # [P, B, H, N] -> [P, B, N, H]  # noqa: E731
    o_ref, l_ref = oracle.lse_combine(o_parts.reshape(P, -1, d), rows(lse_parts).reshape(P, -1))
    o_ref = o_ref.reshape(B, N, H, d)
    l_ref = np.moveaxis(l_ref.reshape(B, N, H), 1, -1)
    o, lse = host(o), host(lse)
    assert np.isfinite(o).all()
    assert (np.abs(o - o_ref) <= 2.0 ** -8 * np.abs(o_ref) + 1e-6).all()
    fin = np.isfinite(l_ref)
    assert np.array_equal(np.isfinite(lse), fin) and (o[1, 7, 2] == 0).all()
    assert np.abs(lse[fin] - l_ref[fin]).max() <= 1e-5


def test_lse_combine_reproduces_the_two_round_example():
    """The two rounds of "FlashAttention：一次前向计算" (figs. 5-10) as two parts
    (d padded from 2 to 64 with zeros): O = [[7/8, 3/4], [4/3, 1/3]], L = ln 8, ln 9."""
    import torch
    g = fixtures.load("p3_two_round_example.txt")
    f = lambda rows: np.array([[float(x) for x in r] for r in rows])  # noqa: E731
    l1 = f([g["l1"]])[0]
    l2 = f(g["P2"]).sum(axis=1)
    parts = np.zeros((2, 1, 2, 1, 64), np.float32)      # [P, B, N, H, d]
    parts[0, 0, :, 0, :2] = f(g["O1"]) / l1[:, None]
    parts[1, 0, :, 0, :2] = f(g["PV2"]) / l2[:, None]
    lse_parts = np.zeros((2, 1, 1, 2), np.float32)
    lse_parts[0, 0, 0] = math.log(2) * f([g["m1"]])[0] + np.log(l1)
    lse_parts[1, 0, 0] = math.log(2) * f([g["m2"]])[0] + np.log(l2)
    o, lse = fa.lse_combine(torch.from_numpy(parts).cuda(), torch.from_numpy(lse_parts).cuda(),
                            dtype=torch.float16)
    o, lse = host(o), host(lse)
    np.testing.assert_allclose(o[0, :, 0, :2], f(g["O"]), atol=2e-3, rtol=0)
    assert (o[0, :, 0, 2:] == 0).all()
    np.testing.assert_allclose(lse[0, 0], [math.log(8), math.log(9)], atol=1e-5, rtol=0)


# --------------------------------------------------------------------------- decoding workload
def test_decode_workload_all_rows():
    w = fa_inputs.WORKLOADS["d1_decode_b8h32kv8nq1nk32768d128"]
    x = fa_inputs.make_workload(w)
    o, lse = run_kv(x["q"], x["k"], x["v"], w.causal, splits=0)
    o_ref, l_ref = oracle.attention(x["q"], x["k"], x["v"], w.scale, w.causal)
    check(o, lse, o_ref, l_ref, w.name)
