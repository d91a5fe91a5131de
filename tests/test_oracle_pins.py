"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test checks the oracle's window (oracle/kda_window.c) against a hand
worked example, a closed form, a special case that reduces to a library
routine, or an independent brute-force formulation, chosen so that a
plausible slip (a dropped term, a wrong sign, a transposed operand, the
norm's eps outside the root, the output taken before the update, decay along
the wrong axis) fails at least one of them.

Source of the definition: the per-token loop of `_verify_kernel` in
recoverssm.py (GLM-5.3-Flash KDA speculative verify) and the gate of kda.py.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import kda_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f(x):
    return float("-inf") if x == "-inf" else float(x)


# ------------------------------------------------------------ worked example

def test_hand_worked_windows():
    with open(os.path.join(GOLDEN, "hand_window.json")) as fh:
        gold = json.load(fh)
    tol = gold["tolerance"]
    for case in gold["cases"]:
        out, traj, h = O.window(
            np.array(case["h0"]), np.array(case["k"]), np.array(case["v"]),
            np.array(case["g_raw"]), np.array(case["beta_raw"]), _f(case["a_log"]),
            np.array(case["g_bias"]), q=np.array(case["q"]), bounded=case["bounded"],
            lower_bound=case["lower_bound"], scale=case["scale"], want_traj=True)
        np.testing.assert_allclose(out, np.array(case["out"]), atol=tol, rtol=0)
        np.testing.assert_allclose(traj, np.array(case["traj"]), atol=tol, rtol=0)
        np.testing.assert_allclose(h, np.array(case["traj"])[-1], atol=tol, rtol=0)


# ------------------------------------------------------------- gate values

def test_gate_special_values():
    # softplus(0) = ln 2, so the default gate at x = 0 is -exp(A_log) ln 2
    for a_log in (0.0, 1.3, -2.0):
        assert O.gate(0.0, a_log, False, 0.0) == pytest.approx(-math.exp(a_log) * math.log(2),
                                                               rel=1e-15)
    # bounded gate: lb * sigmoid(0) = lb / 2, saturates at lb and 0
    assert O.gate(0.0, 0.7, True, -5.0) == pytest.approx(-2.5, rel=1e-15)
    assert O.gate(1e3, 0.0, True, -5.0) == pytest.approx(-5.0, rel=1e-15)
    assert O.gate(-1e3, 0.0, True, -5.0) == pytest.approx(0.0, abs=1e-300)
    # the bounded gate stays inside (lb, 0)
    for x in np.linspace(-30, 30, 61):
        gv = O.gate(x, 0.4, True, -5.0)
        assert -5.0 <= gv <= 0.0
    # the default gate is unbounded below: -a * x for large x
    assert O.gate(30.0, 0.5, False, 0.0) == pytest.approx(-math.exp(0.5) * 30.0, rel=1e-12)
    # and vanishes like -a e^x for very negative x
    assert O.gate(-30.0, 0.0, False, 0.0) == pytest.approx(-math.exp(-30.0), rel=1e-9)


def test_gate_against_library_softplus_and_sigmoid():
    xs = np.linspace(-25, 25, 101)
    for a_log in (-1.0, 0.0, 2.5):
        a = math.exp(a_log)
        ref_soft = -a * torch.nn.functional.softplus(torch.tensor(xs, dtype=torch.float64)).numpy()
        ref_bound = -4.0 * torch.sigmoid(torch.tensor(a * xs, dtype=torch.float64)).numpy()
        got_soft = np.array([O.gate(x, a_log, False, 0.0) for x in xs])
        got_bound = np.array([O.gate(x, a_log, True, -4.0) for x in xs])
        np.testing.assert_allclose(got_soft, ref_soft, rtol=1e-12, atol=1e-300)
        np.testing.assert_allclose(got_bound, ref_bound, rtol=1e-12, atol=1e-300)


# -------------------------------------------------------------- brute force

def _np_gate(x, a_log, bounded, lb):
    a = np.exp(a_log)
    if bounded:
        return lb / (1.0 + np.exp(-a * x))
    return -a * np.logaddexp(0.0, x)


def _unrolled(h0, q, k, v, g_raw, beta_raw, a_log, g_bias, bounded, lb, scale):
    """Transition-matrix form, summed in closed form:
        S_t = S_{t-1} A_t + B_t,  A_t = diag(e_t)(I - b_t kh kh^T),  B_t = b_t v kh^T
        S_T = S_0 A_1..A_T + sum_s B_s A_{s+1}..A_T,  o_t = S_t qh_t."""
    T, K = k.shape
    As, Bs, qs = [], [], []
    for t in range(T):
        kh = k[t] / np.sqrt(k[t] @ k[t] + 1e-6)
        qh = q[t] / np.sqrt(q[t] @ q[t] + 1e-6) * scale
        e = np.exp(_np_gate(g_raw[t] + g_bias, a_log, bounded, lb))
        b = 1.0 / (1.0 + np.exp(-beta_raw[t]))
        As.append(np.diag(e) @ (np.eye(K) - b * np.outer(kh, kh)))
        Bs.append(b * np.outer(v[t], kh))
        qs.append(qh)
    states, outs = [], []
    for t in range(T):
        prod = np.eye(K)
        for r in range(t + 1):
            prod = prod @ As[r]
        S = h0 @ prod
        for s in range(t + 1):
            tail = np.eye(K)
            for r in range(s + 1, t + 1):
                tail = tail @ As[r]
            S = S + Bs[s] @ tail
        states.append(S)
        outs.append(S @ qs[t])
    return np.array(outs), np.array(states)


@pytest.mark.parametrize("K,V,T,bounded", [(2, 3, 3, False), (3, 2, 3, True),
                                           (4, 5, 2, False), (5, 4, 3, True)])
def test_brute_force_unrolled_form(K, V, T, bounded):
    rng = np.random.default_rng(K * 100 + V * 10 + T)
    h0 = rng.normal(size=(V, K))
    q = rng.normal(size=(T, K))
    k = rng.normal(size=(T, K))
    v = rng.normal(size=(T, V))
    g_raw = rng.normal(size=(T, K))
    beta_raw = rng.normal(size=T)
    g_bias = rng.normal(size=K) * 0.3
    a_log, lb, scale = 0.4, -3.0, 0.7
    out, traj, h = O.window(h0, k, v, g_raw, beta_raw, a_log, g_bias, q=q, bounded=bounded,
                            lower_bound=lb, scale=scale, want_traj=True)
    ref_out, ref_states = _unrolled(h0, q, k, v, g_raw, beta_raw, a_log, g_bias, bounded, lb,
                                    scale)
    np.testing.assert_allclose(traj, ref_states, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(out, ref_out, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(h, ref_states[-1], rtol=1e-11, atol=1e-12)


# -------------------------------------------------------------- closed forms

def _rand_token(rng, K=128, V=128):
    return (rng.normal(size=(1, K)), rng.normal(size=(1, K)), rng.normal(size=(1, V)),
            rng.normal(size=(1, K)))


def test_single_token_from_zero():
    # S = beta v kh^T  and  o = beta (kh . qh) v, qh including the scale
    rng = np.random.default_rng(1)
    q, k, v, g = _rand_token(rng)
    braw = np.array([0.3])
    scale = 128 ** -0.5
    out, _, h = O.window(np.zeros((128, 128)), k, v, g, braw, 1.1, rng.normal(size=128) * 0.1,
                         q=q, scale=scale)
    beta = 1.0 / (1.0 + math.exp(-0.3))
    kh = k[0] / math.sqrt(float(k[0] @ k[0]) + 1e-6)
    qh = q[0] / math.sqrt(float(q[0] @ q[0]) + 1e-6) * scale
    np.testing.assert_allclose(h, beta * np.outer(v[0], kh), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(out[0], beta * float(kh @ qh) * v[0], rtol=1e-12, atol=1e-15)


def test_pure_decay_when_beta_vanishes():
    # beta_raw = -1000: sigmoid is exactly 0, so S_T = S_0 diag(exp(sum_t g_t))
    rng = np.random.default_rng(2)
    T, K, V = 4, 128, 128
    h0 = rng.normal(size=(V, K))
    g_raw = rng.normal(size=(T, K))
    bias = rng.normal(size=K) * 0.1
    for bounded, a_log in ((False, 0.9), (True, 0.2)):
        _, _, h = O.window(h0, rng.normal(size=(T, K)), rng.normal(size=(T, V)), g_raw,
                           np.full(T, -1000.0), a_log, bias, bounded=bounded, lower_bound=-5.0)
        gsum = _np_gate(g_raw + bias, a_log, bounded, -5.0).sum(axis=0)
        np.testing.assert_allclose(h, h0 * np.exp(gsum)[None, :], rtol=1e-12, atol=1e-300)


def test_delta_rule_write_without_decay():
    # A_log = -inf: no decay.  beta = 1: after a token, S k^ = (1 - c) S_prev k^ + c v,
    # c = |k|^2 / (|k|^2 + 1e-6) -- the delta rule writes v at key k.
    rng = np.random.default_rng(3)
    h0 = rng.normal(size=(128, 128)) * 0.05
    k = rng.normal(size=(1, 128)) * 1e-3     # small norm: c visibly below 1
    v = rng.normal(size=(1, 128))
    _, _, h = O.window(h0, k, v, rng.normal(size=(1, 128)), np.array([50.0]), float("-inf"),
                       np.zeros(128))
    nk2 = float(k[0] @ k[0])
    c = nk2 / (nk2 + 1e-6)
    kh = k[0] / math.sqrt(nk2 + 1e-6)
    np.testing.assert_allclose(h @ kh, (1 - c) * (h0 @ kh) + c * v[0], rtol=1e-11, atol=1e-13)


def test_norm_eps_inside_root():
    # |k|^2 = 1e-6 exactly scaled: |k^|^2 = 1e-6 / (1e-6 + 1e-6) = 1/2
    k = np.zeros((1, 128))
    k[0, 0] = 1e-3
    v = np.zeros((1, 128))
    v[0, 5] = 2.0
    _, _, h = O.window(np.zeros((128, 128)), k, v, np.zeros((1, 128)), np.array([50.0]),
                       float("-inf"), np.zeros(128))
    # single token from zero, beta = 1: S = v kh^T, S[5, 0] = 2 * kh_0 = 2 / sqrt(2)
    assert h[5, 0] == pytest.approx(2.0 / math.sqrt(2.0), rel=1e-12)


def test_output_is_linear_in_scale_and_invariant_to_q_norm():
    rng = np.random.default_rng(4)
    T = 3
    h0 = rng.normal(size=(128, 128)) * 0.05
    args = (rng.normal(size=(T, 128)), rng.normal(size=(T, 128)), rng.normal(size=(T, 128)),
            rng.normal(size=T), 0.5, rng.normal(size=128) * 0.1)
    q = rng.normal(size=(T, 128))
    o1, _, _ = O.window(h0, *args, q=q, scale=0.25)
    o2, _, _ = O.window(h0, *args, q=q, scale=0.5)
    o3, _, _ = O.window(h0, *args, q=q * 7.0, scale=0.25)
    np.testing.assert_allclose(o2, 2 * o1, rtol=1e-13, atol=1e-16)
    # scaling q by 7 changes q^ only through the eps inside the root
    n2 = (q * q).sum(axis=1)
    ratio = 7.0 * np.sqrt(n2 + 1e-6) / np.sqrt(49.0 * n2 + 1e-6)
    np.testing.assert_allclose(o3, o1 * ratio[:, None], rtol=1e-12, atol=1e-16)
    assert np.abs(ratio - 1).max() > 1e-9   # the eps effect is visible at this size


def test_state_is_affine_in_the_checkpoint():
    # S_T(S_a + S_b) = S_T(S_a) + S_T(S_b) - S_T(0): the recurrence is affine in S_0
    rng = np.random.default_rng(5)
    T = 4
    args = (rng.normal(size=(T, 128)), rng.normal(size=(T, 128)), rng.normal(size=(T, 128)),
            rng.normal(size=T), 1.7, rng.normal(size=128) * 0.1)
    a, b = rng.normal(size=(2, 128, 128))
    _, _, ha = O.window(a, *args)
    _, _, hb = O.window(b, *args)
    _, _, hab = O.window(a + b, *args)
    _, _, h0 = O.window(np.zeros((128, 128)), *args)
    np.testing.assert_allclose(hab, ha + hb - h0, rtol=1e-10, atol=1e-12)


# ----------------------------------------------------------------- rounding

def test_round_bf16_ties_and_library():
    assert O.round_bf16(1.0 + 2 ** -8) == 1.0                  # tie to even
    assert O.round_bf16(1.0 + 3 * 2 ** -8) == 1.0 + 2 ** -6    # tie to even (upward)
    assert O.round_bf16(-(1.0 + 2 ** -8 + 2 ** -20)) == -(1.0 + 2 ** -7)
    rng = np.random.default_rng(6)
    xs = np.concatenate([rng.normal(size=2000), rng.normal(size=2000) * 1e-3])
    lib = torch.tensor(xs, dtype=torch.float64).to(torch.bfloat16).to(torch.float64).numpy()
    mine = np.array([O.round_bf16(x) for x in xs])
    np.testing.assert_array_equal(mine, lib)
