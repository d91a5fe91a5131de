"""GPU parity of the tensor window form, a build option of the library.

With KDA_TENSOR_WINDOW the verify's window items (5 or more new tokens, raw
records, no trajectory output) take their 2T row dot products with the state
on the tensor core: tcgen05.mma of kind::tf32 from a checkpoint staged by a
128-byte-swizzled tensor-map TMA, with each operand split into its TF32 part
and the remainder so that the products keep fp32 accuracy.  The product
library does not enable it (it measured slower than the FMA window form), so
these tests build the variant (build.build_variant) and call it through the
same C ABI.

Checked against the oracle with the output tolerance of test_gpu_parity
(within 2e-3 and within half a bf16 ulp plus 1e-7).  The records and every
stored state are bit-identical to the product library's: the variant changes
only how the outputs are computed.  Items with folded tokens fold token by
token, write the folded state back to the staging buffer and take the same
tensor form.  So a verify after a fold gives the same output bits as a flush
followed by a verify.
"""

import contextlib

import numpy as np
import pytest
import torch

from linear_attention_speculative_kda_gb300 import api
from linear_attention_speculative_kda_gb300 import build as kbuild
from linear_attention_speculative_kda_gb300 import workloads as W
from oracle import kda_oracle as O
from tests.helpers import (DeviceRun, assert_out_close, assert_state_close, oracle_cache,
                           oracle_layer, oracle_step)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tensor_lib():
    return api.bind_library(kbuild.build_variant("tensor_window", ["KDA_TENSOR_WINDOW"]))


@contextlib.contextmanager
def using(lib):
    api.load_library()  # the product library's handle, restored afterwards
    saved = api._lib_handle
    api._lib_handle = lib
    try:
        yield
    finally:
        api._lib_handle = saved


CASES = [
    ("ragged_q8", dict(B=12, H=3, Q=8, lens=[8, 1, 5, 0, 8, 3, 7, 2, 8, 6, 4, 8], S=16, seed=1)),
    ("bounded_q8", dict(B=10, H=2, Q=8, lens=[8, 8, 2, 7, 5, 8, 1, 3, 8, 6], S=13, bounded=True,
                        lower_bound=-5.0, seed=2, slots=[3, 0, 5, 7, 0, 1, 9, 11, 2, 12])),
    ("q5", dict(B=6, H=2, Q=5, lens=[5, 4, 5, 1, 3, 5], S=8, seed=7)),
    ("q7", dict(B=8, H=2, Q=7, lens=[7, 6, 1, 7, 2, 7, 5, 3], S=10, seed=8)),
]


@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_tensor_window_outputs(tensor_lib, name, kw):
    wl = W.custom(**kw)
    g, ref = DeviceRun(wl), DeviceRun(wl)
    with using(tensor_lib):
        g.verify()
        g.commit()
    ref.verify()
    ref.commit()
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0 and int(ref.err.item()) == 0
    assert torch.equal(g.records, ref.records)
    assert torch.equal(g.pool, ref.pool)
    res = O.verify(oracle_layer(wl), oracle_cache(wl), oracle_step(wl))
    assert_out_close(g.out, res.out)
    cu = wl.cu_seqlens.numpy()
    out = g.out.float().cpu().numpy()
    run = set(res.rows_run)
    for b in range(wl.spec.B):
        if b not in run:  # skipped rows keep the sentinel
            assert (out[cu[b]:cu[b + 1]] == -9.0).all()


def test_tensor_window_strong_decay(tensor_lib):
    """Decays down to e^-40 per token (the operands' decay products
    underflow) and beta near 1."""
    wl = W.custom(B=8, H=2, Q=8, lens=[8] * 8, S=10, seed=12)
    wl.A_log[:] = torch.tensor([3.2, 0.1])
    for st in wl.steps:
        st.g_raw.mul_(3.0)
        st.beta_buf.add_(4.0)
    g = DeviceRun(wl)
    with using(tensor_lib):
        g.verify()
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    assert torch.isfinite(g.out.float()).all()
    res = O.verify(oracle_layer(wl), oracle_cache(wl), oracle_step(wl))
    assert_out_close(g.out, res.out)


def test_tensor_window_after_fold_equals_flush(tensor_lib):
    """Window 8, deferred: the second verify folds the pending tokens of some
    rows (tensor form from the folded state) and not of others.  Its outputs
    equal, bit for bit, those of a flush followed by a verify, and the oracle's
    within the tolerance; the folded states equal the product library's."""
    Q = 8
    lens = [Q, Q, 2, Q, 1, Q, Q - 1, Q] * 3
    wl = W.custom(B=len(lens), H=2, Q=Q, lens=lens, S=len(lens) + 6, R=len(lens) + 4,
                  deferred=True, steps=2, seed=48, eager_prob=0.25, bounded=True,
                  lower_bound=-5.0)
    ones = torch.ones_like(wl.steps[1].eager).cuda()
    g, f, ref = DeviceRun(wl), DeviceRun(wl), DeviceRun(wl)
    with using(tensor_lib):
        g.verify(0, pending=True)
        g.commit(0, deferred=True)
        g.verify(1, pending=True)  # folds
        g.commit(1, deferred=True, eager=ones)
        f.verify(0, pending=True)
        f.commit(0, deferred=True)
        f.flush()
        f.verify(1)
        f.commit(1, deferred=True, eager=ones)
    ref.verify(0, pending=True)
    ref.commit(0, deferred=True)
    ref.verify(1, pending=True)
    ref.commit(1, deferred=True, eager=ones)
    torch.cuda.synchronize()
    for r in (g, f, ref):
        assert int(r.err.item()) == 0
    assert torch.equal(g.out, f.out)
    assert torch.equal(g.pool, ref.pool) and torch.equal(f.pool, ref.pool)
    assert torch.equal(g.records, ref.records)
    layer, cache = oracle_layer(wl), oracle_cache(wl)
    s1, s2 = oracle_step(wl, 0), oracle_step(wl, 1)
    O.verify(layer, cache, s1, pending=True)
    O.commit(layer, cache, s1, wl.steps[0].num_accepted.numpy(), deferred=True,
             eager=wl.steps[0].eager.numpy())
    r2 = O.verify(layer, cache, s2, pending=True)
    assert_out_close(g.out, r2.out)


@pytest.mark.parametrize("name", ["dflash7", "mixed"])
def test_tensor_window_full_size_sampled(tensor_lib, name):
    """The full-size window-8 workloads as the benchmark runs them: a sample
    of (row, head) outputs and committed states against the oracle."""
    wl = W.generate(name)
    sp = wl.spec
    g = DeviceRun(wl, sentinel=False)
    with using(tensor_lib):
        g.verify(0, pending=sp.deferred)
        g.commit(0, deferred=sp.deferred)
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    rng = np.random.default_rng(3)
    rows = sorted(rng.choice(sp.B, size=min(sp.B, 24), replace=False).tolist())
    heads = sorted(rng.choice(sp.H, size=min(sp.H, 3), replace=False).tolist())
    layer, step, cache = oracle_layer(wl), oracle_step(wl), oracle_cache(wl)
    res = O.verify(layer, cache, step, pending=sp.deferred, rows=rows, heads=heads)
    acc = wl.steps[0].num_accepted.numpy()
    eager = None if wl.steps[0].eager is None else wl.steps[0].eager.numpy()
    O.commit(layer, cache, step, acc, deferred=sp.deferred, eager=eager, rows=rows, heads=heads)
    assert_out_close(g.out, res.out)
    for (slot, h), ref in cache.written.items():
        assert_state_close(g.pool[slot, h].double().cpu().numpy(), ref)
