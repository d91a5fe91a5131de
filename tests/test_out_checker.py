"""The bf16 output check of the GPU parity tests, exercised on the CPU.

``assert_out_close`` holds every output element to the stated absolute
2e-3 and to half a bf16 ulp of the oracle value plus 1e-7 (what rounding an
fp32 result to bf16 allows).  At these workloads' output scale (median
|o| about 1e-3) the absolute bound alone would pass a result that is
several percent off, so each test here plants a plausible mistake on the
CPU, in the oracle or in the numpy restatement of the window form, and
checks that the checker refuses its bf16-rounded outputs while the stated
bound alone would have passed them.  A correct result, the oracle value
rounded to nearest even, passes.
"""

import numpy as np
import pytest
import torch

from linear_attention_speculative_kda_gb300 import workloads as W
from oracle import kda_oracle as O
from tests.helpers import (OUT_ATOL, assert_out_close, bf16_ulp, oracle_cache, oracle_layer,
                           oracle_step)
from tests.test_window_algebra import _window_form


def _rne(x: np.ndarray) -> np.ndarray:
    """Round to bf16, nearest even (torch's conversion), back to float64."""
    t = torch.from_numpy(np.nan_to_num(x, nan=0.0))
    return t.to(torch.bfloat16).to(torch.float64).numpy()


def _truncate(x: np.ndarray) -> np.ndarray:
    """Round toward zero to bf16 (drop the low 16 bits of the fp32 value)."""
    b = np.nan_to_num(x, nan=0.0).astype(np.float32).view(np.uint32) & np.uint32(0xFFFF0000)
    return b.view(np.float32).astype(np.float64)


def _old_bound_passes(got, ref):
    m = ~np.isnan(ref)
    return np.abs(got[m] - ref[m]).max() <= OUT_ATOL


@pytest.fixture(scope="module")
def case():
    wl = W.custom(B=8, H=2, Q=8, lens=[8, 5, 8, 3, 8, 8, 1, 6], S=12, seed=41)
    layer, step = oracle_layer(wl), oracle_step(wl)
    ref = O.verify(layer, oracle_cache(wl), step).out
    return wl, layer, step, ref


def test_bf16_ulp():
    assert bf16_ulp(1.0) == 2.0 ** -7
    assert bf16_ulp(1.5) == 2.0 ** -7
    assert bf16_ulp(0.999) == 2.0 ** -8
    assert bf16_ulp(-3e-3) == 2.0 ** -16      # 3e-3 in [2^-9, 2^-8)
    # the spacing of adjacent bf16 values, from torch's own rounding
    x = torch.tensor([1e-3, 0.7, 3.0, -40.0], dtype=torch.bfloat16)
    nxt = (x.view(torch.int16) + 1).view(torch.bfloat16)
    np.testing.assert_array_equal(bf16_ulp(x.double().numpy()),
                                  (nxt.double() - x.double()).abs().numpy())


def test_rounded_oracle_passes(case):
    _, _, _, ref = case
    got = _rne(ref)
    assert assert_out_close(got, ref) <= 0.5


def test_truncated_rounding_is_refused(case):
    _, _, _, ref = case
    got = _truncate(ref)
    assert _old_bound_passes(got, ref)
    with pytest.raises(AssertionError, match="bf16 ulp"):
        assert_out_close(got, ref)


@pytest.mark.parametrize("factor", [1.01, 0.99])
def test_scale_error_is_refused(case, factor):
    # a 1% error in the q scale (or in the q norm) scales every output by 1%
    wl, layer, step, ref = case
    bad_layer = O.Layer(layer.num_heads, layer.head_dim, layer.window, layer.a_log,
                        layer.g_bias, layer.bounded, layer.lower_bound, layer.scale * factor)
    got = _rne(O.verify(bad_layer, oracle_cache(wl), step).out)
    assert _old_bound_passes(got, ref)
    with pytest.raises(AssertionError, match="bf16 ulp"):
        assert_out_close(got, ref)


@pytest.mark.parametrize("t,s", [(3, 1), (7, 7), (5, 4), (0, 0)])
def test_window_coefficient_error_is_refused(t, s):
    # one pair coefficient b_ts of the window form off by 2%: the outputs of
    # token t move by 0.02 b_ts v'_s, a few bf16 ulps at this scale
    rng = np.random.default_rng(3)
    T, D = 8, 128
    S = rng.normal(0.0, 0.05, size=(D, D))
    q, k, v, g_raw = (rng.normal(size=(T, D)) for _ in range(4))
    beta_raw, g_bias = rng.normal(size=T), rng.normal(0.0, 0.1, size=D)
    args = (S, q, k, v, g_raw, beta_raw, 1.0, g_bias, False, 0.0, D ** -0.5)
    ref, _, _ = O.window(S, k, v, g_raw, beta_raw, 1.0, g_bias, q=q, scale=D ** -0.5)
    good, _ = _window_form(*args)
    assert_out_close(_rne(good), ref)
    bad, _ = _window_form(*args, perturb_b=(t, s, 1.02))
    got = _rne(bad)
    assert _old_bound_passes(got, ref)
    with pytest.raises(AssertionError, match="bf16 ulp"):
        assert_out_close(got, ref)
