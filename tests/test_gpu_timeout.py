"""The bounded-wait timeout path, on the GPU.

No input of the C ABI can leave one of the kernel's waits unsatisfied, so
this test uses a test build of the library (build.build_variant, compiled
with KDA_TEST_WITHHOLD_END_MARKER and a wait budget of about 10 ms; never
the product library): its producer never tells consumer 0 of CTA 0 that
the work is done.  That consumer's wait for a next item runs out after it
has finished its items, with no copy in flight.  The launch must return,
the error word must carry KDA_ERR_WAIT_TIMEOUT, the outputs must still be
right (every item was processed before the wait), and the product library
must then run correctly in the same process.
"""

import numpy as np
import pytest
import torch

from linear_attention_speculative_kda_gb300 import api
from linear_attention_speculative_kda_gb300 import build as kbuild
from linear_attention_speculative_kda_gb300 import workloads as W
from oracle import kda_oracle as O
from tests.helpers import DeviceRun, assert_out_close, oracle_cache, oracle_layer, oracle_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def starved_lib():
    path = kbuild.build_variant("withhold_end", ["KDA_TEST_WITHHOLD_END_MARKER",
                                                 "KDA_TEST_WAIT_BUDGET=20000000LL"])
    return api.bind_library(path)


def _verify_with(lib, g):
    saved = api._lib_handle
    api._lib_handle = lib
    try:
        g.verify()
    finally:
        api._lib_handle = saved


def test_wait_timeout_is_reported_and_the_context_stays_usable(starved_lib):
    wl = W.generate("tiny")
    g = DeviceRun(wl)
    _verify_with(starved_lib, g)
    torch.cuda.synchronize()                          # the launch returns
    assert int(g.err.item()) == api.ERR_WAIT_TIMEOUT
    res = O.verify(oracle_layer(wl), oracle_cache(wl), oracle_step(wl))
    assert_out_close(g.out, res.out)                  # the items ran before the wait
    # the product library, in the same process, afterwards
    h = DeviceRun(wl)
    h.verify()
    h.commit()
    torch.cuda.synchronize()
    assert int(h.err.item()) == 0
    assert_out_close(h.out, res.out)
    assert torch.equal(h.out, g.out)


def test_a_second_starved_launch_times_out_again(starved_lib):
    wl = W.custom(B=10, H=3, Q=8, lens=[8, 3, 8, 5, 1, 8, 0, 7, 8, 2], S=14, seed=71)
    g = DeviceRun(wl)
    for _ in range(2):
        g.err.zero_()
        _verify_with(starved_lib, g)
        torch.cuda.synchronize()
        assert int(g.err.item()) == api.ERR_WAIT_TIMEOUT
    assert torch.equal(g.pool, g.pool0)
