"""GPU: independent calls on two streams at once give the sequential bits.

The library keeps no device-side global state and its kernels never wait on
one another, so two workloads' verify / commit sequences issued on two
streams, their launches free to overlap, must leave exactly what each leaves
when run alone on the default stream.
"""

import pytest
import torch

from linear_attention_speculative_kda_gb300 import workloads as W
from tests.helpers import DeviceRun

pytestmark = pytest.mark.gpu


def _issue(g, deferred):
    if deferred:
        g.verify(0, pending=True)
        g.commit(0, deferred=True)
        g.verify(1, pending=True)
        g.commit(1, deferred=True)
    else:
        g.verify(0)
        g.commit(0)


def test_two_streams_match_sequential_runs():
    wa = W.custom(B=96, H=8, Q=4, lens=[4, 3, 4, 2] * 24, S=110, R=100, deferred=True, steps=2,
                  seed=61, eager_prob=0.3)
    wb = W.custom(B=64, H=8, Q=8, lens=[8, 5, 2, 8] * 16, S=70, seed=62, bounded=True,
                  lower_bound=-5.0)
    ref_a, ref_b = DeviceRun(wa), DeviceRun(wb)
    _issue(ref_a, True)
    _issue(ref_b, False)
    torch.cuda.synchronize()
    a, b = DeviceRun(wa), DeviceRun(wb)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    sa.wait_stream(torch.cuda.current_stream())
    sb.wait_stream(torch.cuda.current_stream())
    # both sequences are queued before either finishes: their launches may overlap
    with torch.cuda.stream(sa):
        _issue(a, True)
    with torch.cuda.stream(sb):
        _issue(b, False)
    torch.cuda.synchronize()
    for got, want in ((a, ref_a), (b, ref_b)):
        assert int(got.err.item()) == 0
        assert torch.equal(got.out, want.out)
        assert torch.equal(got.records, want.records)
        assert torch.equal(got.pool, want.pool)
        assert torch.equal(got.pending, want.pending)
