"""Invariants of the oracle's verify / commit / flush bookkeeping.

These are the properties the pages state for RecoverSSM:
- the committed state after n accepted tokens is the state the full-state
  path stores after token n (recoverssm.py module docstring and the commit's
  replay comment);
- accepting 0 tokens, or a null state index, writes nothing
  (`_prepare_commit_plan_kernel`, `_verify_kernel`);
- the deferred commit (Kimi-K3 context page) reaches the same states and
  outputs as committing eagerly, and flush gives a non-folding verify the
  same start.
"""

import numpy as np
import torch

from linear_attention_speculative_kda_gb300 import workloads as W
from oracle import kda_oracle as O
from tests.helpers import oracle_cache, oracle_layer, oracle_step


def _tiny(**kw):
    base = dict(B=5, H=2, Q=4, lens=[4, 3, 0, 4, 1], S=9, seed=11)
    base.update(kw)
    return W.custom(**base)


def test_commit_equals_trajectory_state():
    wl = _tiny()
    layer, step = oracle_layer(wl), oracle_step(wl)
    cache = oracle_cache(wl)
    res = O.verify(layer, cache, step, want_traj=True)
    assert not cache.written            # verify never stores a state
    acc = np.array([3, 2, 4, 0, 1])
    O.commit(layer, cache, step, acc)
    for b in range(wl.spec.B):
        T = int(step.cu_seqlens[b + 1] - step.cu_seqlens[b])
        n = O.commit_len(acc[b], T, layer.window)
        slot = int(step.state_indices[b])
        for h in range(layer.num_heads):
            if n == 0:
                assert (slot, h) not in cache.written
            else:
                tok = int(step.cu_seqlens[b]) + n - 1
                np.testing.assert_array_equal(cache.written[(slot, h)], res.traj[(tok, h)])


def test_commit_plan_clamps():
    assert O.commit_len(-3, 4, 4) == 0
    assert O.commit_len(7, 3, 4) == 3
    assert O.commit_len(7, 8, 4) == 4
    assert O.commit_len(2, 4, 4) == 2


def test_null_and_empty_rows_are_skipped():
    wl = _tiny(slots=[3, 0, 5, 0, 7])
    layer, step = oracle_layer(wl), oracle_step(wl)
    cache = oracle_cache(wl)
    res = O.verify(layer, cache, step)
    assert sorted(res.rows_run) == [0, 4]      # row 2 has T == 0, rows 1, 3 are null
    cu = step.cu_seqlens
    for b in (1, 3):
        assert np.isnan(res.out[cu[b]:cu[b + 1]]).all()
    assert {r for (r, _) in cache.records} == {0, 4}
    O.commit(layer, cache, step, np.array([4, 4, 4, 4, 4]))
    assert {s for (s, _) in cache.written} == {3, 7}


def test_row_permutation_equivariance():
    wl = _tiny()
    layer, step = oracle_layer(wl), oracle_step(wl)
    res = O.verify(layer, oracle_cache(wl), step)
    perm = np.array([3, 0, 4, 2, 1])
    cu = step.cu_seqlens
    toks = np.concatenate([np.arange(cu[b], cu[b + 1]) for b in perm]).astype(int)
    lens = (cu[1:] - cu[:-1])[perm]
    cu_p = np.concatenate([[0], np.cumsum(lens)])
    step_p = O.Step(q=step.q[toks], k=step.k[toks], v=step.v[toks], g_raw=step.g_raw[toks],
                    beta_raw=step.beta_raw[toks], cu_seqlens=cu_p,
                    state_indices=step.state_indices[perm], record_rows=None)
    res_p = O.verify(layer, oracle_cache(wl), step_p)
    np.testing.assert_array_equal(res_p.out, res.out[toks])


def _two_steps(deferred: bool, eager_mask, acc1, acc2, use_flush=False):
    wl = W.custom(B=6, H=2, Q=4, lens=[4, 4, 2, 4, 3, 4], S=10, R=8, deferred=True, steps=2,
                  seed=21)
    layer = oracle_layer(wl)
    cache = oracle_cache(wl)
    s1, s2 = oracle_step(wl, 0), oracle_step(wl, 1)
    r1 = O.verify(layer, cache, s1, pending=deferred)
    O.commit(layer, cache, s1, acc1, deferred=deferred, eager=eager_mask if deferred else None)
    if use_flush:
        O.flush(layer, cache, s2)
        r2 = O.verify(layer, cache, s2, pending=False)
    else:
        r2 = O.verify(layer, cache, s2, pending=deferred)
    O.commit(layer, cache, s2, acc2)
    return r1, r2, cache


def test_deferred_two_steps_equal_eager_two_steps():
    acc1 = np.array([2, 0, 2, 4, 1, 3])
    acc2 = np.array([4, 1, 1, 3, 3, 0])
    eager = np.array([0, 0, 1, 0, 0, 1], np.uint8)
    e1, e2, ce = _two_steps(False, None, acc1, acc2)
    d1, d2, cd = _two_steps(True, eager, acc1, acc2)
    f1, f2, cf = _two_steps(True, eager, acc1, acc2, use_flush=True)
    np.testing.assert_array_equal(e1.out, d1.out)
    np.testing.assert_array_equal(e2.out, d2.out)
    np.testing.assert_array_equal(e2.out, f2.out)
    assert ce.written.keys() == cd.written.keys() == cf.written.keys()
    for key in ce.written:
        np.testing.assert_array_equal(ce.written[key], cd.written[key])
        np.testing.assert_array_equal(ce.written[key], cf.written[key])


def test_deferred_commit_sets_pending():
    wl = W.custom(B=4, H=1, Q=4, lens=[4, 4, 4, 0], S=8, R=6, deferred=True,
                  record_rows=[5, -1, 2, 0], slots=[1, 2, 0, 3], seed=3)
    layer, step = oracle_layer(wl), oracle_step(wl)
    cache = oracle_cache(wl)
    cache.pending[:] = 9                      # stale values
    O.verify(layer, cache, step)
    O.commit(layer, cache, step, np.array([3, 2, 4, 1]), deferred=True,
             eager=np.array([0, 0, 0, 0], np.uint8))
    # row 0 valid: pending 3; row 1 has no record slot: nothing written;
    # row 2 is null: pending 0; row 3 has T == 0 so n == 0: pending 0
    assert cache.pending.tolist() == [0, 9, 0, 9, 9, 3]
    assert not cache.written


def test_invalid_rows_are_reported():
    wl = W.custom(B=4, H=1, Q=4, lens=[4, 4, 4, 4], S=4, seed=5, slots=[1, 2, 3, 1])
    layer = oracle_layer(wl)
    step = oracle_step(wl, cu_seqlens=torch.tensor([0, 4, 9, 12, 16], dtype=torch.int32),
                       state_indices=torch.tensor([1, 2, 9, 3], dtype=torch.int32),
                       record_rows=np.array([0, 1, 2, 7]))
    cache = oracle_cache(wl)
    res = O.verify(layer, cache, step)
    # row 1: T = 5 > Q; row 2: slot 9 >= S = 4; row 3: record slot 7 >= R = 4
    assert {i.row: i.reason for i in res.issues} == {1: "length", 2: "slot", 3: "record"}
    assert res.rows_run == [0]
    cache.pending[0] = 5                       # > Q: invalid pending count
    res = O.verify(layer, cache, step, pending=True, rows=[0])
    assert [(i.row, i.reason) for i in res.issues] == [(0, "pending")]


def test_deferred_commit_clears_pending_of_skipped_rows():
    # rows skipped for bad metadata still have their pending count rewritten
    # (to 0) when their record slot is usable: the slot's records were just
    # overwritten by this step's verify, so an old count would replay them
    wl = W.custom(B=4, H=1, Q=4, lens=[4, 4, 4, 4], S=6, R=6, deferred=True,
                  record_rows=[1, 2, 3, 4], slots=[1, 2, 3, 4], seed=9)
    layer = oracle_layer(wl)
    step = oracle_step(wl, cu_seqlens=torch.tensor([0, 4, 9, 12, 16], dtype=torch.int32),
                       state_indices=torch.tensor([1, 2, 9, 3], dtype=torch.int32),
                       record_rows=np.array([1, 2, 3, 8]))
    cache = oracle_cache(wl)
    cache.pending[:] = 3                      # stale counts of the previous step
    issues = O.commit(layer, cache, step, np.array([2, 2, 2, 2]), deferred=True,
                      eager=np.zeros(4, np.uint8))
    # row 1: T = 5 > Q; row 2: slot 9 >= S; row 3: record slot 8 >= R (not written)
    assert {i.row: i.reason for i in issues} == {1: "length", 2: "slot", 3: "record"}
    assert cache.pending.tolist() == [3, 2, 0, 0, 3, 3]
