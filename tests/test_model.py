"""Pins for the CPU model of the blocked update (oracle/online_softmax.py)."""
import math

import numpy as np
import pytest

import fa_inputs
import oracle
from oracle.online_softmax import online_softmax_rows
from tests.golden import fixtures


def f(rows):
    return np.array([[float(x) for x in r] for r in rows], dtype=np.float64)


def test_p3_round_by_round_states():
    """tau = 0 is the standard online softmax; its states match figures 5-10 of the page."""
    g = fixtures.load("p3_two_round_example.txt")
    o, lse, st = online_softmax_rows(f(g["Q"]), f(g["K"]), f(g["V"]), scale_log2=1.0, block_n=2,
                                     tau=0.0, reverse=False, trace=True)
    assert len(st) == 2
    np.testing.assert_array_equal(st[0]["ref"], [float(x) for x in g["m1"]])
    np.testing.assert_array_equal(st[0]["row_sum"], [float(x) for x in g["l1"]])
    np.testing.assert_array_equal(st[0]["O"], f(g["O1"]))
    np.testing.assert_array_equal(st[1]["acc_scale"], [float(x) for x in g["alpha2"]])
    np.testing.assert_array_equal(st[1]["ref"], [float(x) for x in g["m2"]])
    np.testing.assert_array_equal(st[1]["row_sum"], [float(x) for x in g["l2"]])
    np.testing.assert_array_equal(st[1]["O"], f(g["O2"]))
    np.testing.assert_allclose(o, f(g["O"]), atol=1e-15, rtol=0)
    np.testing.assert_allclose(lse, [math.log(float(x)) for x in g["LSE_ln"]], atol=1e-15, rtol=0)


@pytest.mark.parametrize("case", ["A", "B"])
def test_p1_exercise1_threshold_rule(case):
    ex = fixtures.load("p1_exercises.txt")
    r0, l0, o0, o1 = (float(x) for x in ex["EX1_STATE"])
    s = np.array([[float(x) for x in ex[f"EX1_{case}_S"]]])
    ref, acc, rs, w0, w1 = (float(x) for x in ex[f"EX1_{case}_OUT"])
    # one query row, two keys; q = [1, 0] and k rows = [S0, 0], [S1, 0] produce the scores S
    q = np.array([[1.0, 0.0]])
    k = np.array([[s[0, 0], 0.0], [s[0, 1], 0.0]])
    v = np.eye(2)
    _, _, st = online_softmax_rows(q, k, v, scale_log2=1.0, block_n=2, tau=8.0,
                                   init=([r0], [l0], [[o0, o1]]), trace=True)
    assert st[0]["ref"][0] == ref
    assert st[0]["acc_scale"][0] == acc
    assert st[0]["row_sum"][0] == rs
    np.testing.assert_array_equal(st[0]["O"][0], [w0, w1])
    # and O / row_sum equals the direct softmax over (old keys at reference 2) + new keys
    direct_num = np.array([o0, o1]) * 2.0 ** (r0 - ref) + 2.0 ** (s[0] - ref) @ v
    direct_den = l0 * 2.0 ** (r0 - ref) + (2.0 ** (s[0] - ref)).sum()
    np.testing.assert_allclose(st[0]["O"][0] / st[0]["row_sum"][0], direct_num / direct_den, rtol=1e-15)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("tau", [0.0, 8.0, 1e30])
def test_result_does_not_depend_on_tau(causal, tau):
    N, d = 300, 64
    q, k, v = fa_inputs.make_qkv(1, N, 1, d, seed=50, spiky=True)
    o_ref, l_ref = oracle.attention(q, k, v, 1 / math.sqrt(d), causal)
    qf, kf, vf = (fa_inputs.bf16_bits_to_f32(x)[0, :, 0].astype(np.float64) for x in (q, k, v))
    sl2 = math.log2(math.e) / math.sqrt(d)
    for row0 in (0, 128, 256):
        rows = slice(row0, min(row0 + 128, N))
        o, lse = online_softmax_rows(qf[rows], kf, vf, scale_log2=sl2, block_n=128, tau=tau,
                                     causal=causal, row0=row0)
        np.testing.assert_allclose(o, o_ref[0, rows, 0], atol=1e-12, rtol=0)
        np.testing.assert_allclose(lse, l_ref[0, 0, rows], atol=1e-12, rtol=0)


def test_rescale_fires_on_spiky_inputs():
    """The spiky recipe makes the reference jump by more than tau within a row."""
    N, d = 2048, 128
    q, k, v = fa_inputs.make_qkv(1, N, 1, d, seed=20264, spiky=True)
    qf, kf, vf = (fa_inputs.bf16_bits_to_f32(x)[0, :, 0].astype(np.float64) for x in (q, k, v))
    sl2 = math.log2(math.e) / math.sqrt(d)
    _, _, st = online_softmax_rows(qf[1920:2048], kf, vf, scale_log2=sl2, block_n=128, tau=8.0,
                                   causal=True, row0=1920, trace=True)
    fired = sum(int((s["acc_scale"] < 1).sum()) for s in st[1:])
    assert fired > 0


def test_bf16_p_and_fp32_state_stay_within_tolerance():
    """fp32 state plus bf16 rounding of P (what the kernel does) stays inside O 2e-2 / LSE 1e-3."""
    N, d = 512, 128
    q, k, v = fa_inputs.make_qkv(1, N, 1, d, seed=51, spiky=True)
    o_ref, l_ref = oracle.attention(q, k, v, 1 / math.sqrt(d), True)
    qf, kf, vf = (fa_inputs.bf16_bits_to_f32(x)[0, :, 0] for x in (q, k, v))
    sl2 = math.log2(math.e) / math.sqrt(d)
    for row0 in range(0, N, 128):
        o, lse = online_softmax_rows(qf[row0:row0 + 128], kf, vf, scale_log2=sl2, block_n=128,
                                     tau=8.0, causal=True, row0=row0, dtype=np.float32,
                                     p_round="bf16")
        assert np.abs(o - o_ref[0, row0:row0 + 128, 0]).max() < 2e-2
        assert np.abs(lse - l_ref[0, 0, row0:row0 + 128]).max() < 1e-3
