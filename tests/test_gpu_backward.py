"""GPU parity for the backward pass (fa_bwd) against the fp64 oracle gradients.

The forward runs on the GPU first (it supplies O and the LSE the backward
reuses); the oracle differentiates the exact definition from the same 16-bit
inputs. Tolerance: the gradients pass through three 16-bit roundings (P for dV,
dS for dQ and dK, and the outputs), each a relative 2^-9 (bf16) of terms of the
size of the gradient; the bound is max |grad - oracle| <= 2e-2 * max(1, max |oracle|)
per tensor, the forward's O tolerance scaled by the gradient's magnitude.
"""
import math

import numpy as np
import pytest

import attention_forward_tma_gb300 as fa
import fa_inputs
import oracle

pytestmark = pytest.mark.gpu

TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.library()
    yield torch


def tdtype(dtype):
    import torch
    return torch.float16 if dtype == "f16" else torch.bfloat16


def dev(bits, dtype="bf16"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(tdtype(dtype)).cuda()


def host(t):
    import torch
    dtype = "f16" if t.dtype == torch.float16 else "bf16"
    return fa_inputs.bits_to_f32(t.view(torch.int16).cpu().numpy().view(np.uint16), dtype).astype(np.float64)


def run_bwd(q, k, v, do, causal, dtype="bf16", scale=None):
    qd, kd, vd, dod = dev(q, dtype), dev(k, dtype), dev(v, dtype), dev(do, dtype)
    o, lse = fa.fa_fwd(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = fa.fa_bwd(qd, kd, vd, o, dod, lse, causal=causal, scale=scale)
    st, word = fa.last_device_status()
    assert st == fa.FA_OK, hex(word)
    return host(dq), host(dk), host(dv)


def check(got, ref, what):
    errs = []
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        assert np.isfinite(g).all(), f"{what}: non-finite {name}"
        bound = TOL * max(1.0, np.abs(r).max())
        err = np.abs(g - r).max()
        errs.append(f"{name} {err:.2e}/{bound:.2e}")
        assert err <= bound, f"{what}: max |{name} - oracle| = {err} > {bound}"
    print(what, " ".join(errs))


SHAPES = [  # (B, H, H_kv, N_q, N_kv, d)
    (1, 1, 1, 128, 128, 128),
    (1, 2, 2, 300, 300, 128),
    (2, 4, 1, 129, 129, 64),      # multi-query, ragged
    (1, 8, 2, 200, 333, 128),     # G = 4, N_q < N_kv
    (1, 4, 4, 100, 257, 64),
    (1, 32, 1, 40, 40, 64),       # G = 32
    (1, 2, 2, 257, 100, 128),     # N_q > N_kv: causal rows without keys
    (1, 1, 1, 640, 640, 128),     # several key blocks and Q tiles
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%dH%dKV%dNq%dNk%dd%d" % s)
def test_backward_elementwise(shape, causal):
    B, H, Hkv, Nq, Nk, d = shape
    q, k, v = fa_inputs.make_qkv(B, Nq, H, d, seed=4000 + Nq + Nk + H, Nkv=Nk, Hkv=Hkv)
    do = fa_inputs.make_qkv(B, Nq, H, d, seed=5000 + Nq)[0]
    got = run_bwd(q, k, v, do, causal)
    ref = oracle.attention_backward(q, k, v, do, 1 / math.sqrt(d), causal)
    check(got, ref, f"{shape} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_backward_fp16(causal):
    q, k, v = fa_inputs.make_qkv(1, 300, 8, 128, seed=4100, Hkv=2, dtype="f16")
    do = fa_inputs.make_qkv(1, 300, 8, 128, seed=4101, dtype="f16")[0]
    got = run_bwd(q, k, v, do, causal, "f16")
    ref = oracle.attention_backward(q, k, v, do, 1 / math.sqrt(128), causal, dtype="f16")
    check(got, ref, f"fp16 causal={causal}")


def test_backward_spiky_scores():
    q, k, v = fa_inputs.make_qkv(1, 400, 2, 128, seed=20264, spiky=True)
    do = fa_inputs.make_qkv(1, 400, 2, 128, seed=4200)[0]
    got = run_bwd(q, k, v, do, True)
    ref = oracle.attention_backward(q, k, v, do, 1 / math.sqrt(128), True)
    check(got, ref, "spiky")


def test_backward_dk_dv_deterministic():
    q, k, v = fa_inputs.make_qkv(1, 500, 4, 128, seed=4300, Hkv=2)
    do = fa_inputs.make_qkv(1, 500, 4, 128, seed=4301)[0]
    a = run_bwd(q, k, v, do, True)
    b = run_bwd(q, k, v, do, True)
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
    assert np.abs(a[0] - b[0]).max() <= 2.0 ** -7 * max(1.0, np.abs(a[0]).max())


@pytest.mark.parametrize("shape", [(1, 4, 2, 500, 500, 128, True), (2, 8, 1, 300, 700, 64, False),
                                   (1, 2, 2, 900, 900, 128, False)],
                         ids=lambda s: "B%dH%dKV%dNq%dNk%dd%d_causal%d" % s)
def test_backward_deterministic_mode(shape):
    """With bwd_deterministic set, the key blocks add their dQ contributions in
    key-block order: two runs give bitwise-equal dQ, and parity holds."""
    B, H, Hkv, Nq, Nk, d, causal = shape
    q, k, v = fa_inputs.make_qkv(B, Nq, H, d, seed=4400 + Nq, Nkv=Nk, Hkv=Hkv)
    do = fa_inputs.make_qkv(B, Nq, H, d, seed=4401 + Nq)[0]
    fa.set_option("bwd_deterministic", 1)
    try:
        a = run_bwd(q, k, v, do, causal)
        b = run_bwd(q, k, v, do, causal)
    finally:
        fa.set_option("bwd_deterministic", 0)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    check(a, oracle.attention_backward(q, k, v, do, 1 / math.sqrt(d), causal), f"deterministic {shape}")


# --------------------------------------------------------------------------- varlen
def run_bwd_varlen(lq, lk, H, Hkv, d, causal, dtype="bf16", seed=0):
    """Packed sequences (query lengths lq, key lengths lk) through fa_fwd_varlen and
    fa_bwd_varlen; returns the inputs, cu arrays and host gradients."""
    import torch
    rng = np.random.default_rng(seed)
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    T, Tk = int(cu_q[-1]), int(cu_k[-1])
    f = lambda shape: fa_inputs.f32_to_bits(rng.standard_normal(shape).astype(np.float32), dtype)  # noqa: E731
    q, k, v, do = f((T, H, d)), f((Tk, Hkv, d)), f((Tk, Hkv, d)), f((T, H, d))
    cq, ck = torch.from_numpy(cu_q).cuda(), torch.from_numpy(cu_k).cuda()
    qd, kd, vd, dod = dev(q, dtype), dev(k, dtype), dev(v, dtype), dev(do, dtype)
    o, lse = fa.fa_fwd_varlen(qd, kd, vd, cq, max(lq), cu_seqlens_k=ck, max_seqlen_k=max(lk), causal=causal)
    dq, dk, dv = fa.fa_bwd_varlen(qd, kd, vd, o, dod, lse, cq, max(lq), cu_seqlens_k=ck, max_seqlen_k=max(lk),
                                  causal=causal)
    st, word = fa.last_device_status()
    assert st == fa.FA_OK, hex(word)
    return (q, k, v, do, cu_q, cu_k), (host(dq), host(dk), host(dv))


VARLEN = [  # (query lengths, key lengths, H, H_kv, d)
    ([7, 0, 129, 300, 1, 520], None, 4, 2, 128),
    ([200, 64, 333], [250, 64, 100], 8, 2, 128),     # N_q != N_kv per sequence (causal rows without keys)
    ([130, 5, 260], [0, 40, 300], 2, 1, 64),          # a sequence without keys
    ([40, 90], None, 32, 1, 64),                       # G = 32
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("case", VARLEN, ids=lambda c: f"q{c[0]}_k{c[1]}_H{c[2]}KV{c[3]}d{c[4]}")
def test_backward_varlen_elementwise(case, causal):
    lq, lk, H, Hkv, d = case
    lk = lq if lk is None else lk
    (q, k, v, do, cu_q, cu_k), got = run_bwd_varlen(lq, lk, H, Hkv, d, causal, seed=sum(lq) + H)
    ref = oracle.attention_backward_varlen(q, k, v, do, cu_q, cu_k, 1 / math.sqrt(d), causal)
    check(got, ref, f"varlen {lq}/{lk} causal={causal}")


def test_backward_varlen_fp16_and_deterministic():
    lq = [300, 17, 450]
    fa.set_option("bwd_deterministic", 1)
    try:
        (q, k, v, do, cu_q, cu_k), a = run_bwd_varlen(lq, lq, 8, 2, 128, True, "f16", seed=9)
        _, b = run_bwd_varlen(lq, lq, 8, 2, 128, True, "f16", seed=9)
    finally:
        fa.set_option("bwd_deterministic", 0)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    ref = oracle.attention_backward_varlen(q, k, v, do, cu_q, cu_k, 1 / math.sqrt(128), True, dtype="f16")
    check(a, ref, "varlen fp16 deterministic")


# --------------------------------------------------------------------------- full sizes
def _full_inputs(name):
    """A named workload's inputs and the upstream gradient bench.py draws for it."""
    w = fa_inputs.WORKLOADS[name]
    x = fa_inputs.make_workload(w)
    if w.varlen:
        T = x["q"].shape[0]
        do = fa_inputs.make_qkv(1, T, w.H, w.d, w.seed + 1000, dtype=w.dtype)[0][0]
    else:
        do = fa_inputs.make_qkv(w.B, w.N, w.H, w.d, w.seed + 1000, dtype=w.dtype)[0]
    return w, x, do


@pytest.mark.parametrize("name,b,kvh", [("c3_b4h16n4096d128_causal", 2, 11),
                                        ("g2_gqa_b4h32kv8n4096d128_causal", 3, 5)])
def test_backward_full_size_one_head_group(name, b, kvh):
    """The whole workload through the kernel in bench.py's launch configuration; the
    gradients of one (batch, K/V head) group checked in full against the oracle on that
    group alone (its dK, dV and its query heads' dQ depend on nothing else)."""
    w, x, do = _full_inputs(name)
    got = run_bwd(x["q"], x["k"], x["v"], do, w.causal, w.dtype, scale=w.scale)
    G = w.H // w.Hkv
    hs = slice(kvh * G, (kvh + 1) * G)
    q, k, v = x["q"][b:b + 1, :, hs], x["k"][b:b + 1, :, kvh:kvh + 1], x["v"][b:b + 1, :, kvh:kvh + 1]
    ref = oracle.attention_backward(q, k, v, do[b:b + 1, :, hs], w.scale, w.causal, dtype=w.dtype)
    sel = (got[0][b:b + 1, :, hs], got[1][b:b + 1, :, kvh:kvh + 1], got[2][b:b + 1, :, kvh:kvh + 1])
    check(sel, ref, f"{name} b={b} kv head={kvh}")
    for g in got:   # every other gradient at least finite
        assert np.isfinite(g).all()


def test_backward_full_size_every_element():
    """c3 (B4 H16 N4096 d128 causal) through the kernel in bench.py's launch
    configuration: every element of dQ, dK and dV against the fp64 oracle."""
    w, x, do = _full_inputs("c3_b4h16n4096d128_causal")
    got = run_bwd(x["q"], x["k"], x["v"], do, w.causal, w.dtype, scale=w.scale)
    ref = oracle.attention_backward(x["q"], x["k"], x["v"], do, w.scale, w.causal, dtype=w.dtype)
    check(got, ref, f"c3 full: {got[0].size} dQ, {got[1].size} dK and {got[2].size} dV elements")


def test_backward_full_size_varlen_one_sequence():
    import torch
    w, x, do = _full_inputs("c5_varlen8_h16d128_causal")
    cu = x["cu_seqlens"]
    qd, kd, vd, dod = dev(x["q"]), dev(x["k"]), dev(x["v"]), dev(do)
    cd = torch.from_numpy(cu).cuda()
    maxL = int(x["lengths"].max())
    o, lse = fa.fa_fwd_varlen(qd, kd, vd, cd, maxL, scale=w.scale, causal=True)
    dq, dk, dv = fa.fa_bwd_varlen(qd, kd, vd, o, dod, lse, cd, maxL, scale=w.scale, causal=True)
    st, word = fa.last_device_status()
    assert st == fa.FA_OK, hex(word)
    s = int(np.argmax(x["lengths"]))          # the longest sequence, one head
    a, e, h = int(cu[s]), int(cu[s + 1]), 9
    ref = oracle.attention_backward(x["q"][None, a:e, h:h + 1], x["k"][None, a:e, h:h + 1],
                                    x["v"][None, a:e, h:h + 1], do[None, a:e, h:h + 1], w.scale, True)
    got = tuple(host(t)[None, a:e, h:h + 1] for t in (dq, dk, dv))
    check(got, ref, f"c5 sequence {s} (length {e - a}) head {h}")


def test_backward_full_size_deterministic_bits():
    w, x, do = _full_inputs("c3_b4h16n4096d128_causal")
    fa.set_option("bwd_deterministic", 1)
    try:
        a = run_bwd(x["q"], x["k"], x["v"], do, True, scale=w.scale)
        b = run_bwd(x["q"], x["k"], x["v"], do, True, scale=w.scale)
    finally:
        fa.set_option("bwd_deterministic", 0)
    for g, h in zip(a, b):
        assert np.array_equal(g, h)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_scheduling_modes_agree(causal):
    """Persistent CTAs claiming tasks against one CTA per task, and L2 sections of
    different sizes: dK and dV (accumulated in tensor memory in a fixed order) are
    bitwise equal; dQ (added across key blocks in arrival order) agrees within the
    tolerance."""
    q, k, v = fa_inputs.make_qkv(2, 700, 8, 128, seed=4500, Hkv=2)
    do = fa_inputs.make_qkv(2, 700, 8, 128, seed=4501)[0]
    runs = []
    for persistent, section in ((-1, 0), (0, 0), (-1, 1), (-1, 3)):
        fa.set_option("persistent", persistent)
        fa.set_option("bwd_section", section)
        try:
            runs.append(run_bwd(q, k, v, do, causal))
        finally:
            fa.set_option("persistent", -1)
            fa.set_option("bwd_section", 0)
    ref = oracle.attention_backward(q, k, v, do, 1 / math.sqrt(128), causal)
    for got in runs:
        assert np.array_equal(got[1], runs[0][1]) and np.array_equal(got[2], runs[0][2])
        check(got, ref, f"scheduling causal={causal}")
