"""GPU parity of the verify's window form: in a raw-record verify without a
trajectory output, each item with at least 5 new tokens computes their
outputs from the starting state in one set of row dot products and a
per-row triangular solve, instead of token by token (the state is not
updated; the commit replays as before); shorter items stay token by token.
The small cases with Q >= 5 here mix both kinds of items in one launch
(rows of 1 to Q tokens); those with Q <= 4 check that nothing changes for
them; the full-size ones run as the benchmark runs them.

Tolerances, as in test_gpu_parity: bf16 outputs within 2e-3 of the oracle
and within half a bf16 ulp of it plus 1e-7 (the window form rounds its
fp32 outputs like the token-by-token form, so the same bound holds);
records and every stored state (the fold's, the commit's) bit-identical to
the token-by-token run, which is itself bit-checked against its trajectory.
"""

import numpy as np
import pytest
import torch

from linear_attention_speculative_kda_gb300 import workloads as W
from oracle import kda_oracle as O
from tests.helpers import (DeviceRun, assert_out_close, assert_state_close, oracle_cache,
                           oracle_layer, oracle_step)

pytestmark = pytest.mark.gpu


def _cases():
    yield "ragged_q8", W.custom(B=12, H=3, Q=8, lens=[8, 1, 5, 0, 8, 3, 7, 2, 8, 6, 4, 8],
                                S=16, seed=1)
    yield "bounded_q8", W.custom(B=10, H=2, Q=8, lens=[8, 8, 2, 7, 5, 8, 1, 3, 8, 6], S=13,
                                 bounded=True, lower_bound=-5.0, seed=2,
                                 slots=[3, 0, 5, 7, 0, 1, 9, 11, 2, 12])
    yield "q1", W.custom(B=6, H=4, Q=1, lens=[1, 1, 0, 1, 1, 1], S=8, seed=3)
    yield "q2", W.custom(B=7, H=2, Q=2, lens=[2, 1, 2, 2, 0, 2, 1], S=9, seed=5)
    yield "q3", W.custom(B=7, H=2, Q=3, lens=[3, 1, 2, 3, 3, 0, 2], S=9, seed=6)
    yield "q5", W.custom(B=6, H=2, Q=5, lens=[5, 4, 5, 1, 3, 5], S=8, seed=7)
    yield "q7", W.custom(B=8, H=2, Q=7, lens=[7, 6, 1, 7, 2, 7, 5, 3], S=10, seed=8)
    yield "q4", W.custom(B=9, H=2, Q=4, lens=[4, 4, 2, 4, 0, 3, 4, 1, 4], S=12, seed=4)


CASES = list(_cases())


@pytest.mark.parametrize("name,wl", CASES, ids=[c[0] for c in CASES])
def test_window_outputs_records_and_commit(name, wl):
    gw = DeviceRun(wl)                        # window form (no trajectory output)
    gs = DeviceRun(wl, with_traj=True)        # token by token
    for g in (gw, gs):
        g.verify()
        g.commit()
    torch.cuda.synchronize()
    assert int(gw.err.item()) == 0 and int(gs.err.item()) == 0
    assert torch.equal(gw.records, gs.records)
    assert torch.equal(gw.pool, gs.pool)
    layer, step = oracle_layer(wl), oracle_step(wl)
    res = O.verify(layer, oracle_cache(wl), step)
    assert_out_close(gw.out, res.out)
    # rows the verify skipped keep the sentinel
    cu = wl.cu_seqlens.numpy()
    run = set(res.rows_run)
    out = gw.out.float().cpu().numpy()
    for b in range(wl.spec.B):
        if b not in run:
            assert (out[cu[b]:cu[b + 1]] == -9.0).all()


def test_window_strong_decay_and_large_beta():
    """Gates near their extremes (decays down to e^-40 per token, so the
    window's decay products underflow) and beta near 1."""
    wl = W.custom(B=8, H=2, Q=8, lens=[8] * 8, S=10, seed=12)
    wl.A_log[:] = torch.tensor([3.2, 0.1])
    for st in wl.steps:
        st.g_raw.mul_(3.0)
        st.beta_buf.add_(4.0)
    gw = DeviceRun(wl)
    gw.verify()
    torch.cuda.synchronize()
    assert int(gw.err.item()) == 0
    assert torch.isfinite(gw.out.float()).all()
    res = O.verify(oracle_layer(wl), oracle_cache(wl), oracle_step(wl))
    assert_out_close(gw.out, res.out)


@pytest.mark.parametrize("Q,bounded", [(4, False), (8, True)])
def test_window_after_fold(Q, bounded):
    lens = [Q, Q, 2, Q, 1, Q, Q - 1, 0] * 3
    kw = dict(bounded=True, lower_bound=-5.0) if bounded else {}
    wl = W.custom(B=len(lens), H=2, Q=Q, lens=lens, S=len(lens) + 6, R=len(lens) + 4,
                  deferred=True, steps=2, seed=60 + Q, eager_prob=0.25, **kw)
    gw, gs = DeviceRun(wl), DeviceRun(wl, with_traj=True)
    for g in (gw, gs):
        g.verify(0, pending=True)
        g.commit(0, deferred=True)
        g.verify(1, pending=True)
    torch.cuda.synchronize()
    assert int(gw.err.item()) == 0 and int(gs.err.item()) == 0
    assert torch.equal(gw.pool, gs.pool)          # the folded states
    assert torch.equal(gw.records, gs.records)
    layer = oracle_layer(wl)
    cache = oracle_cache(wl)
    s1, s2 = oracle_step(wl, 0), oracle_step(wl, 1)
    O.verify(layer, cache, s1, pending=True)
    O.commit(layer, cache, s1, wl.steps[0].num_accepted.numpy(), deferred=True,
             eager=wl.steps[0].eager.numpy())
    r2 = O.verify(layer, cache, s2, pending=True)
    assert_out_close(gw.out, r2.out)
    pool = gw.pool.cpu()
    for (slot, h), ref in cache.written.items():
        assert_state_close(pool[slot, h].double().numpy(), ref)


@pytest.mark.parametrize("name", ["mtp3", "dflash7", "mixed", "deferred2"])
def test_full_size_window_sampled(name):
    """The full-size workloads in the benchmark's launch configuration
    (window form for dflash7's items and mixed's longer ones, token by token
    otherwise): a sample of (row, head) outputs and committed states
    against the oracle."""
    wl = W.generate(name)
    sp = wl.spec
    deferred = sp.deferred
    g = DeviceRun(wl, sentinel=False)
    g.verify(0, pending=deferred)
    g.commit(0, deferred=deferred)
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    rng = np.random.default_rng(1)
    rows = sorted(rng.choice(sp.B, size=min(sp.B, 24), replace=False).tolist())
    heads = sorted(rng.choice(sp.H, size=min(sp.H, 3), replace=False).tolist())
    layer, step = oracle_layer(wl), oracle_step(wl)
    cache = oracle_cache(wl)
    res = O.verify(layer, cache, step, pending=deferred, rows=rows, heads=heads)
    acc = wl.steps[0].num_accepted.numpy()
    eager = None if wl.steps[0].eager is None else wl.steps[0].eager.numpy()
    O.commit(layer, cache, step, acc, deferred=deferred, eager=eager, rows=rows, heads=heads)
    assert_out_close(g.out, res.out)
    for (slot, h), ref in cache.written.items():
        assert_state_close(g.pool[slot, h].double().cpu().numpy(), ref)


def test_window_strided_activations_eight_byte_aligned():
    """Window form with activation rows whose token stride is a multiple of
    4 elements but not of 8, starting 8 bytes past a 16-byte boundary: the
    same bits as the packed layout."""
    from linear_attention_speculative_kda_gb300 import api
    wl = W.custom(B=9, H=3, Q=8, lens=[8, 3, 0, 8, 5, 1, 8, 7, 6], S=12, seed=23)
    ref = DeviceRun(wl)
    ref.verify()
    g = DeviceRun(wl)
    st = g.steps[0]
    T, H, D = st["qkv"].shape[0], wl.spec.H, wl.spec.D
    width = 3 * H * D + 4
    flat = torch.zeros(T * width + 4, dtype=torch.bfloat16, device="cuda")
    view = flat[4:].view(T, width)
    view[:, : 3 * H * D] = st["qkv"].reshape(T, -1)
    q = view[:, 0 * H * D:1 * H * D].view(T, H, D)
    k = view[:, 1 * H * D:2 * H * D].view(T, H, D)
    v = view[:, 2 * H * D:3 * H * D].view(T, H, D)
    assert q.stride(0) % 8 == 4 and q.data_ptr() % 16 == 8
    api.kda_verify(q, k, v, st["g_raw"], st["beta_buf"][:, :H], g.A_log, g.g_bias, g.pool, g.cu,
                   g.slots, g.records, g.out, error_word=g.err, **g.kw())
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0 and int(ref.err.item()) == 0
    assert torch.equal(g.out, ref.out)
    assert torch.equal(g.records, ref.records)
    res = O.verify(oracle_layer(wl), oracle_cache(wl), oracle_step(wl))
    assert_out_close(g.out, res.out)


def test_window_kernel_error_word_and_skips():
    """Bad metadata in a launch of the window kernel (window 8): the bad rows
    are flagged and skipped, the others run in window form."""
    from linear_attention_speculative_kda_gb300 import api
    wl = W.custom(B=5, H=2, Q=8, lens=[8, 8, 8, 8, 8], S=8, R=6, seed=13,
                  slots=[1, 2, 3, 4, 5], record_rows=[0, 1, 2, 3, 4])
    g = DeviceRun(wl)
    cu = torch.tensor([0, 8, 17, 24, 32, 40], dtype=torch.int32, device="cuda")  # row 1: T = 9
    slots = torch.tensor([1, 2, 11, 4, 5], dtype=torch.int32, device="cuda")     # row 2: 11 >= S
    rr = torch.tensor([0, 1, 2, 9, 4], dtype=torch.int32, device="cuda")         # row 3: 9 >= R
    g.verify(cu=cu, slots=slots, record_rows=rr)
    torch.cuda.synchronize()
    assert int(g.err.item()) == api.ROW_BAD_LENGTH | api.ROW_BAD_SLOT | api.ROW_BAD_RECORD
    out = g.out.float().cpu().numpy()
    assert (out[8:32] == -9.0).all()            # rows 1..3 skipped
    assert not (out[0:8] == -9.0).any()         # rows 0 and 4 ran
    assert not (out[32:40] == -9.0).any()
    assert torch.equal(g.pool, g.pool0)


def test_window_rows_without_record_slot():
    """Rows whose record slot is -1 verify in window form into the scratch
    row and are never committed."""
    wl = W.custom(B=6, H=2, Q=8, lens=[8, 8, 6, 8, 5, 8], S=10, R=6, deferred=True, seed=31,
                  record_rows=[0, -1, 2, -1, 4, 5])
    g = DeviceRun(wl)
    g.verify(pending=True)
    g.commit(deferred=True, eager=torch.ones(6, dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    layer, step = oracle_layer(wl), oracle_step(wl)
    cache = oracle_cache(wl)
    res = O.verify(layer, cache, step, pending=True)
    O.commit(layer, cache, step, wl.steps[0].num_accepted.numpy(), deferred=True,
             eager=np.ones(6, np.uint8))
    assert_out_close(g.out, res.out)
    slots = wl.state_indices.numpy()
    for b in (1, 3):
        assert torch.equal(g.pool[int(slots[b])], g.pool0[int(slots[b])])
    pool = g.pool.cpu()
    for (slot, h), ref in cache.written.items():
        assert_state_close(pool[slot, h].double().numpy(), ref)
