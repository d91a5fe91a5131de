"""The algebra of the verify's window form, in double precision on the CPU.

The window form computes a verify's new-token outputs from the starting
state S without updating it: with G_t = e_1 ... e_t and r_st = e_{s+1} ...
e_t (per channel),
    w_t = S (G_t * k^_t),   y_t = S (G_t * q^_t),
    a_ts = sum_c k^_s r_st k^_t  (s < t),   b_ts = sum_c k^_s r_st q^_t  (s <= t),
    v'_t = beta_t (v_t - w_t - sum_{s<t} a_ts v'_s),
    o_t  = y_t + sum_{s<=t} b_ts v'_s.
These formulas are restated here in numpy and checked against the oracle's
token-by-token recurrence, so a wrong index, a missing decay or a dropped
term in the derivation fails on the CPU.  (The CUDA kernels are checked
against the oracle on the GPU in test_gpu_window.)
"""

import numpy as np
import pytest

from oracle import kda_oracle as O


def _np_gate(x, a_log, bounded, lb):
    a = np.exp(a_log)
    if bounded:
        return lb / (1.0 + np.exp(-a * x))
    return -a * np.logaddexp(0.0, x)


def _window_form(S, q, k, v, g_raw, beta_raw, a_log, g_bias, bounded, lb, scale,
                 perturb_b=None):
    # perturb_b = (t, s, factor): multiplies b_ts by factor (a planted
    # mistake, for the tests of the output checker)
    T = k.shape[0]
    kh = k / np.sqrt((k * k).sum(axis=1, keepdims=True) + 1e-6)
    qh = q / np.sqrt((q * q).sum(axis=1, keepdims=True) + 1e-6) * scale
    e = np.exp(_np_gate(g_raw + g_bias, a_log, bounded, lb))
    beta = 1.0 / (1.0 + np.exp(-beta_raw))
    G = np.cumprod(e, axis=0)
    w = (S @ (G * kh).T).T          # [T, V]
    y = (S @ (G * qh).T).T
    a = np.zeros((T, T))
    b = np.zeros((T, T))
    for s in range(T):
        r = np.ones(k.shape[1])
        for t in range(s, T):
            if t > s:
                r = r * e[t]
                a[t, s] = np.sum(kh[s] * r * kh[t])
            b[t, s] = np.sum(kh[s] * r * qh[t])
    if perturb_b is not None:
        b[perturb_b[0], perturb_b[1]] *= perturb_b[2]
    vp = np.zeros_like(v)
    out = np.zeros_like(v)
    for t in range(T):
        vp[t] = beta[t] * (v[t] - w[t] - sum(a[t, s] * vp[s] for s in range(t)))
        out[t] = y[t] + sum(b[t, s] * vp[s] for s in range(t + 1))
    return out, vp


@pytest.mark.parametrize("T,K,V,bounded", [(1, 128, 128, False), (4, 128, 128, False),
                                           (8, 128, 128, True), (5, 16, 24, False),
                                           (8, 32, 8, True)])
def test_window_form_equals_the_recurrence(T, K, V, bounded):
    rng = np.random.default_rng(100 + T + K)
    S = rng.normal(size=(V, K)) * 0.3
    q, k = rng.normal(size=(T, K)), rng.normal(size=(T, K))
    v, g_raw = rng.normal(size=(T, V)), rng.normal(size=(T, K))
    beta_raw, g_bias = rng.normal(size=T), rng.normal(size=K) * 0.1
    a_log, lb, scale = 1.1, -5.0, K ** -0.5
    out_w, vp_w = _window_form(S, q, k, v, g_raw, beta_raw, a_log, g_bias, bounded, lb, scale)
    out_r, _, _, vp_r = O.window_deltas(S, k, v, g_raw, beta_raw, a_log, g_bias, q=q,
                                        bounded=bounded, lower_bound=lb, scale=scale)
    np.testing.assert_allclose(vp_w, vp_r, rtol=0, atol=1e-11)
    np.testing.assert_allclose(out_w, out_r, rtol=0, atol=1e-11)


def test_window_form_with_vanishing_decay():
    # gates of about -40 per token: the decay products underflow towards 0,
    # and the outputs still match the recurrence (the state is forgotten)
    rng = np.random.default_rng(7)
    T, K, V = 8, 128, 128
    S = rng.normal(size=(V, K))
    q, k = rng.normal(size=(T, K)), rng.normal(size=(T, K))
    v = rng.normal(size=(T, V))
    g_raw = rng.normal(size=(T, K)) * 3.0 + 10.0
    beta_raw = rng.normal(size=T)
    out_w, _ = _window_form(S, q, k, v, g_raw, beta_raw, 2.0, np.zeros(K), False, 0.0,
                            K ** -0.5)
    out_r, _, _ = O.window(S, k, v, g_raw, beta_raw, 2.0, np.zeros(K), q=q, scale=K ** -0.5)
    np.testing.assert_allclose(out_w, out_r, rtol=0, atol=1e-11)
