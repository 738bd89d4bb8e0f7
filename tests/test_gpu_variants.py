"""GPU parity of the forward's tuning variants ("Flash Attention 4", section on the
differences between the paper and the TIRx kernel): the two softmax warpgroups
taking turns at their exponential phases (softmax_stagger) and the rescale
factor passed through tensor memory (stats_tmem).

The default is stats_tmem = 1, softmax_stagger = 0. Both options change only how
the warpgroups synchronise, not the arithmetic, so every combination must give
the default path's bits exactly, and match the fp64 oracle
within the forward's tolerance (O <= 2e-2, LSE <= 1e-3 max-abs). The shapes cover
the cases where the turn count differs between the tiles: causal tasks whose
tile 0 skips the top key block, tasks with a single tile, grouped heads, key
lengths other than the query length, and variable-length batches.
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
VARIANTS = [(0, 0), (1, 0), (1, 1)]   # (softmax_stagger, stats_tmem); default (0, 1)


@pytest.fixture(scope="module", autouse=True)
def cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.library()
    yield torch
    fa.set_option("softmax_stagger", 0)
    fa.set_option("stats_tmem", 1)


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


def with_variant(variant, run):
    stagger, stats = variant
    fa.set_option("softmax_stagger", stagger)
    fa.set_option("stats_tmem", stats)
    try:
        out = run()
    finally:
        fa.set_option("softmax_stagger", 0)
        fa.set_option("stats_tmem", 1)
    return out


def run_fixed(q, k, v, causal):
    o, lse = fa.fa_fwd(dev(q), dev(k), dev(v), causal=causal)
    st, word = fa.last_device_status()
    assert st == fa.FA_OK, hex(word)
    return host(o), host(lse)


def check(o, lse, o_ref, lse_ref, what):
    assert np.isfinite(o).all(), what
    err_o = np.abs(o - o_ref).max()
    assert err_o <= TOL_O, f"{what}: max |O - oracle| = {err_o}"
    fin = np.isfinite(lse_ref)
    assert (np.isneginf(lse) == ~fin).all(), what
    err_l = np.abs(lse[fin] - lse_ref[fin]).max() if fin.any() else 0.0
    assert err_l <= TOL_LSE, f"{what}: max |LSE - oracle| = {err_l}"


SHAPES = [  # (B, H, H_kv, N_q, N_kv, d, spiky)
    (1, 2, 2, 1100, 1100, 128, True),     # causal tile 0 skips the top block; rescales fire
    (2, 3, 3, 700, 700, 64, False),
    (1, 2, 2, 100, 100, 128, False),      # one tile per task
    (1, 8, 2, 300, 300, 128, False),      # grouped heads, G = 4
    (1, 4, 1, 200, 650, 128, False),      # N_q < N_kv
    (1, 2, 2, 650, 200, 128, False),      # N_q > N_kv: causal rows without keys
]


@pytest.mark.parametrize("variant", VARIANTS, ids=lambda v: "stagger%d_tmem%d" % v)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%dH%dKV%dNq%dNk%dd%d_spiky%d" % s)
def test_variant_matches_default_and_oracle(shape, causal, variant):
    B, H, Hkv, Nq, Nk, d, spiky = shape
    if spiky:
        q, k, v = fa_inputs.make_qkv(B, Nq, H, d, seed=20264, spiky=True)
    else:
        q, k, v = fa_inputs.make_qkv(B, Nq, H, d, seed=6000 + Nq + Nk + H, Nkv=Nk, Hkv=Hkv)
    base = run_fixed(q, k, v, causal)
    got = with_variant(variant, lambda: run_fixed(q, k, v, causal))
    assert np.array_equal(base[0], got[0]) and np.array_equal(base[1], got[1]), "differs from the default path"
    o_ref, l_ref = oracle.attention(q, k, v, 1 / math.sqrt(d), causal)
    check(got[0], got[1], o_ref, l_ref, f"{shape} causal={causal} variant={variant}")


@pytest.mark.parametrize("variant", VARIANTS, ids=lambda v: "stagger%d_tmem%d" % v)
def test_variant_varlen(variant):
    import torch
    lengths = [7, 0, 129, 300, 1, 520]
    _, cu, q, k, v = fa_inputs.make_varlen_from_lengths(lengths, 4, 128, seed=6100, Hkv=2)
    cu_d = torch.from_numpy(cu).cuda()

    def run():
        o, lse = fa.fa_fwd_varlen(dev(q), dev(k), dev(v), cu_d, max(lengths), causal=True)
        st, word = fa.last_device_status()
        assert st == fa.FA_OK, hex(word)
        return host(o), host(lse)

    base = run()
    got = with_variant(variant, run)
    assert np.array_equal(base[0], got[0]) and np.array_equal(base[1], got[1])
    o_ref, l_ref = oracle.attention_varlen(q, k, v, cu, 1 / math.sqrt(128), True)
    check(got[0], got[1], o_ref, l_ref, f"varlen variant={variant}")
