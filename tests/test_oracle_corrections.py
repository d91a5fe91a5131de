"""Pins of the oracle's correction-record path (the fp32-correction commit of
the Kimi-K3 deferred context page: the verify records each token's k, g_raw
and delta v' = beta (v - S k^), and the commit folds the deltas into the
checkpoint in closed form).

The closed form is checked against things other than itself: the
recurrence it unrolls (the oracle window, pinned in test_oracle_pins), a
plain matrix product when nothing decays, a pure product of decays when
every delta is zero, and the deltas recomputed by numpy from the window's
own trajectory.
"""

import numpy as np
import pytest

from linear_attention_speculative_kda_gb300 import workloads as W
from oracle import kda_oracle as O
from tests.helpers import oracle_layer, oracle_step


def _np_gate(x, a_log, bounded, lb):
    a = np.exp(a_log)
    if bounded:
        return lb / (1.0 + np.exp(-a * x))
    return -a * np.logaddexp(0.0, x)


def _np_khat(k):
    return k / np.sqrt((k * k).sum(axis=-1, keepdims=True) + 1e-6)


def _inputs(rng, T, K, V):
    return dict(h0=rng.normal(size=(V, K)) * 0.3, k=rng.normal(size=(T, K)),
                v=rng.normal(size=(T, V)), g_raw=rng.normal(size=(T, K)),
                beta_raw=rng.normal(size=T), g_bias=rng.normal(size=K) * 0.1)


@pytest.mark.parametrize("bounded", [False, True])
def test_deltas_match_numpy_on_the_trajectory(bounded):
    # each recorded delta is beta_t (v_t - (S_{t-1} diag(e_t)) k^_t), and
    # S_t = S_{t-1} diag(e_t) + delta_t k^_t^T, recomputed here in numpy from
    # the window's trajectory
    rng = np.random.default_rng(7)
    T, K, V, a_log = 4, 5, 3, 0.4
    x = _inputs(rng, T, K, V)
    _, traj, _, delta = O.window_deltas(x["h0"], x["k"], x["v"], x["g_raw"], x["beta_raw"],
                                        a_log, x["g_bias"], bounded=bounded, lower_bound=-4.0,
                                        want_traj=True)
    kh = _np_khat(x["k"])
    e = np.exp(_np_gate(x["g_raw"] + x["g_bias"], a_log, bounded, -4.0))
    beta = 1.0 / (1.0 + np.exp(-x["beta_raw"]))
    prev = x["h0"]
    for t in range(T):
        dec = prev * e[t][None, :]
        want = beta[t] * (x["v"][t] - dec @ kh[t])
        np.testing.assert_allclose(delta[t], want, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(traj[t], dec + np.outer(want, kh[t]), rtol=1e-12, atol=1e-14)
        prev = traj[t]


@pytest.mark.parametrize("bounded,n", [(False, 1), (False, 3), (True, 4), (False, 8)])
def test_closed_form_equals_the_recurrence(bounded, n):
    # folding the deltas of the first n tokens reaches the window's state
    # after token n (a wrong decay index or a dropped term fails this)
    rng = np.random.default_rng(10 + n)
    K = V = 128
    x = _inputs(rng, 8, K, V)
    _, traj, _, delta = O.window_deltas(x["h0"], x["k"], x["v"], x["g_raw"], x["beta_raw"],
                                        1.3, x["g_bias"], bounded=bounded, lower_bound=-5.0,
                                        want_traj=True)
    h = O.fold_deltas(x["h0"], x["k"][:n], x["g_raw"][:n], delta[:n], 1.3, x["g_bias"],
                      bounded=bounded, lower_bound=-5.0)
    scale = np.abs(traj[n - 1]).max()
    np.testing.assert_allclose(h, traj[n - 1], rtol=0, atol=1e-12 * scale)


def test_closed_form_without_decay_is_a_matrix_product():
    # A_log = -inf: exp(A_log) = 0, every gate is 0 and nothing decays, so
    # the fold is S_0 + D^T K^ (deltas D, normalised keys K^)
    rng = np.random.default_rng(4)
    n, K, V = 5, 128, 128
    h0 = rng.normal(size=(V, K))
    k = rng.normal(size=(n, K))
    d = rng.normal(size=(n, V))
    h = O.fold_deltas(h0, k, rng.normal(size=(n, K)), d, float("-inf"), rng.normal(size=K))
    np.testing.assert_allclose(h, h0 + d.T @ _np_khat(k), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("bounded", [False, True])
def test_closed_form_with_zero_deltas_is_pure_decay(bounded):
    rng = np.random.default_rng(5)
    n, K, V, a_log = 4, 128, 96, 0.7
    h0 = rng.normal(size=(V, K))
    g_raw = rng.normal(size=(n, K))
    bias = rng.normal(size=K) * 0.1
    h = O.fold_deltas(h0, rng.normal(size=(n, K)), g_raw, np.zeros((n, V)), a_log, bias,
                      bounded=bounded, lower_bound=-3.0)
    gsum = _np_gate(g_raw + bias, a_log, bounded, -3.0).sum(axis=0)
    np.testing.assert_allclose(h, h0 * np.exp(gsum)[None, :], rtol=1e-12, atol=1e-300)


def test_closed_form_of_no_tokens_is_the_checkpoint():
    h0 = np.arange(12.0).reshape(3, 4)
    h = O.fold_deltas(h0, np.zeros((0, 4)), np.zeros((0, 4)), np.zeros((0, 3)), 0.5,
                      np.zeros(4))
    np.testing.assert_array_equal(h, h0)


def _two_steps(fmt, eager_mask, acc1, acc2, use_flush=False):
    wl = W.custom(B=6, H=2, Q=4, lens=[4, 4, 2, 4, 3, 4], S=10, R=8, deferred=True, steps=2,
                  seed=21)
    layer = oracle_layer(wl)
    cache = O.Cache(wl.pool.numpy(), wl.spec.record_slots, record_format=fmt)
    s1, s2 = oracle_step(wl, 0), oracle_step(wl, 1)
    r1 = O.verify(layer, cache, s1, pending=True)
    O.commit(layer, cache, s1, acc1, deferred=True, eager=eager_mask)
    if use_flush:
        O.flush(layer, cache, s2)
        r2 = O.verify(layer, cache, s2, pending=False)
    else:
        r2 = O.verify(layer, cache, s2, pending=True)
    O.commit(layer, cache, s2, acc2)
    return r1, r2, cache


@pytest.mark.parametrize("use_flush", [False, True])
def test_correction_records_reach_the_raw_states(use_flush):
    # the deferred protocol with correction records (commit, fold in the next
    # verify, flush) gives the raw-record replay's outputs and states
    acc1 = np.array([2, 0, 2, 4, 1, 3])
    acc2 = np.array([4, 1, 1, 3, 3, 0])
    eager = np.array([0, 0, 1, 0, 0, 1], np.uint8)
    a1, a2, ca = _two_steps("raw", eager, acc1, acc2, use_flush)
    c1, c2, cc = _two_steps("correction", eager, acc1, acc2, use_flush)
    np.testing.assert_array_equal(a1.out, c1.out)
    np.testing.assert_allclose(c2.out, a2.out, rtol=0, atol=1e-12)
    assert ca.written.keys() == cc.written.keys()
    for key in ca.written:
        np.testing.assert_allclose(cc.written[key], ca.written[key], rtol=0, atol=1e-12)


def test_correction_records_hold_k_g_and_delta():
    wl = W.custom(B=2, H=1, Q=4, lens=[3, 4], S=4, seed=8)
    layer, step = oracle_layer(wl), oracle_step(wl)
    cache = O.Cache(wl.pool.numpy(), wl.spec.record_slots, record_format="correction")
    O.verify(layer, cache, step)
    rec = cache.records[(0, 0)]
    np.testing.assert_array_equal(rec["k"][:3], step.k[0:3, 0])
    np.testing.assert_array_equal(rec["g"][:3], step.g_raw[0:3, 0])
    _, _, _, delta = O.window_deltas(cache.state(int(step.state_indices[0]), 0), step.k[0:3, 0],
                                     step.v[0:3, 0], step.g_raw[0:3, 0], step.beta_raw[0:3, 0],
                                     layer.a_log[0], layer.g_bias[0], q=step.q[0:3, 0],
                                     scale=layer.scale)
    np.testing.assert_array_equal(rec["delta"][:3], delta)
    with pytest.raises(ValueError):
        O.Cache(wl.pool.numpy(), 2, record_format="fp8")
