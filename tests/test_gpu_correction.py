"""GPU parity of the correction-record format (the fp32-correction commit of
the Kimi-K3 deferred context): the verify records each token's fp32 delta
v' with its bf16 k and g_raw, and the commit, the deferred fold and the
flush apply the deltas without the prediction S k^.

Tolerances, as in test_gpu_parity:
- bf16 outputs: |gpu - oracle| <= 2e-3 element by element, and within half a
  bf16 ulp of the oracle value plus 1e-7;
- fp32 states: normwise per tile, max |gpu - oracle| <= 1e-5 * max |oracle|;
- recorded deltas: per (row, head, token) vector, max |gpu - oracle| <=
  1e-5 * max(1, max |oracle|) (a delta is a difference of O(1) values);
- recorded k and g_raw: bit-identical copies of the inputs;
- states: bit-identical to the raw-record path (the same operations in the
  same order after v'), and committed states bit-identical to the verify
  trajectory; outputs: the correction format's verify runs token by token,
  the raw format's production verify in window form, so they agree to the
  output tolerance, not bit for bit.
"""

import numpy as np
import pytest
import torch

from linear_attention_speculative_kda_gb300 import api
from linear_attention_speculative_kda_gb300 import workloads as W
from oracle import kda_oracle as O
from tests.helpers import (DeviceRun, assert_out_close, assert_state_close, oracle_cache,
                           oracle_layer, oracle_step)

pytestmark = pytest.mark.gpu

CB = api.CORRECTION_RECORD_BYTES


def _records(g):
    """Correction records as (delta fp32 [R+1, H, Q, 128], k bf16, g_raw bf16)."""
    sp = g.wl.spec
    raw = g.records.view(torch.uint8).reshape(sp.record_slots + 1, sp.H, sp.Q, CB).cpu()
    delta = raw[..., :512].contiguous().view(torch.float32)
    k = raw[..., 512:768].contiguous().view(torch.bfloat16)
    gr = raw[..., 768:].contiguous().view(torch.bfloat16)
    return delta, k, gr


def _cases():
    yield "ragged_q8", W.custom(B=12, H=3, Q=8, lens=[8, 1, 5, 0, 8, 3, 7, 2, 8, 6, 4, 8],
                                S=16, seed=1)
    yield "bounded_q8", W.custom(B=10, H=2, Q=8, lens=[8, 8, 2, 7, 5, 8, 1, 3, 8, 6], S=13,
                                 bounded=True, lower_bound=-5.0, seed=2,
                                 slots=[3, 0, 5, 7, 0, 1, 9, 11, 2, 12])
    yield "q1", W.custom(B=6, H=4, Q=1, lens=[1, 1, 0, 1, 1, 1], S=8, seed=3)
    yield "q4", W.custom(B=9, H=2, Q=4, lens=[4, 4, 2, 4, 0, 3, 4, 1, 4], S=12, seed=4)


CASES = list(_cases())


@pytest.mark.parametrize("name,wl", CASES, ids=[c[0] for c in CASES])
def test_verify_records_deltas(name, wl):
    gr, gc = DeviceRun(wl), DeviceRun(wl, record_format="correction")
    gr.verify()
    gc.verify()
    torch.cuda.synchronize()
    assert int(gr.err.item()) == 0 and int(gc.err.item()) == 0
    assert torch.equal(gc.pool, gc.pool0)          # a verify without pending stores no state
    layer, step = oracle_layer(wl), oracle_step(wl)
    cache = oracle_cache(wl, "correction")
    res = O.verify(layer, cache, step)
    assert_out_close(gc.out, res.out)
    assert_out_close(gr.out, res.out)
    delta, k, g_raw = _records(gc)
    cu = wl.cu_seqlens.numpy()
    st = wl.steps[0]
    for b in res.rows_run:
        T = cu[b + 1] - cu[b]
        for h in range(wl.spec.H):
            assert torch.equal(k[b + 1, h, :T], st.k[cu[b]:cu[b + 1], h])
            assert torch.equal(g_raw[b + 1, h, :T], st.g_raw[cu[b]:cu[b + 1], h])
            ref = cache.records[(b, h)]["delta"][:T]
            err = np.abs(delta[b + 1, h, :T].double().numpy() - ref).max(axis=1)
            lim = 1e-5 * np.maximum(1.0, np.abs(ref).max(axis=1))
            assert (err <= lim).all(), (b, h, err.max())


@pytest.mark.parametrize("name,wl", CASES, ids=[c[0] for c in CASES])
def test_commit_bit_equal_to_raw_and_trajectory(name, wl):
    gr = DeviceRun(wl)
    gc = DeviceRun(wl, record_format="correction", with_traj=True)
    for g in (gr, gc):
        g.verify()
        g.commit()
    torch.cuda.synchronize()
    assert int(gr.err.item()) == 0 and int(gc.err.item()) == 0
    assert torch.equal(gr.pool, gc.pool)
    acc = wl.steps[0].num_accepted.numpy()
    cu = wl.cu_seqlens.numpy()
    for b in range(wl.spec.B):
        slot = int(wl.state_indices[b])
        n = O.commit_len(int(acc[b]), cu[b + 1] - cu[b], wl.spec.Q)
        if slot > 0 and n > 0:
            assert torch.equal(gc.pool[slot], gc.traj[int(cu[b]) + n - 1])
        elif slot > 0:
            assert torch.equal(gc.pool[slot], gc.pool0[slot])
    layer, step = oracle_layer(wl), oracle_step(wl)
    cache = oracle_cache(wl, "correction")
    O.verify(layer, cache, step)
    assert O.commit(layer, cache, step, acc) == []
    pool = gc.pool.cpu().numpy()
    for (slot, h), ref in cache.written.items():
        assert_state_close(pool[slot, h].astype(np.float64), ref)


@pytest.mark.parametrize("Q,bounded", [(4, False), (8, True)])
def test_deferred_fold_and_flush(Q, bounded):
    lens = [Q, Q, 2, Q, 1, Q, Q - 1, Q] * 3
    kw = dict(bounded=True, lower_bound=-5.0) if bounded else {}
    wl = W.custom(B=len(lens), H=2, Q=Q, lens=lens, S=len(lens) + 6, R=len(lens) + 4,
                  deferred=True, steps=2, seed=40 + Q, eager_prob=0.25, **kw)
    ones = torch.ones_like(wl.steps[1].eager).cuda()
    runs = {}
    for fmt in ("raw", "correction"):
        g = DeviceRun(wl, record_format=fmt)
        g.verify(0, pending=True)
        g.commit(0, deferred=True)
        g.verify(1, pending=True)                   # folds the pending deltas
        g.commit(1, deferred=True, eager=ones)
        f = DeviceRun(wl, record_format=fmt)           # the same with a flush instead of a fold
        f.verify(0, pending=True)
        f.commit(0, deferred=True)
        f.flush()
        f.verify(1)
        f.commit(1, deferred=True, eager=ones)
        runs[fmt] = (g, f)
    torch.cuda.synchronize()
    (gr, fr), (gc, fc) = runs["raw"], runs["correction"]
    for g in (gr, fr, gc, fc):
        assert int(g.err.item()) == 0
    assert torch.equal(gc.out, fc.out) and torch.equal(gr.out, fr.out)
    assert torch.equal(gr.pool, gc.pool) and torch.equal(gc.pool, fc.pool)
    assert torch.equal(fr.pool, fc.pool)
    layer = oracle_layer(wl)
    cache = oracle_cache(wl, "correction")
    s1, s2 = oracle_step(wl, 0), oracle_step(wl, 1)
    O.verify(layer, cache, s1, pending=True)
    O.commit(layer, cache, s1, wl.steps[0].num_accepted.numpy(), deferred=True,
             eager=wl.steps[0].eager.numpy())
    r2 = O.verify(layer, cache, s2, pending=True)
    O.commit(layer, cache, s2, wl.steps[1].num_accepted.numpy())
    assert_out_close(gc.out, r2.out)
    assert_out_close(gr.out, r2.out)
    pool = gc.pool.cpu()
    for (slot, h), ref in cache.written.items():
        assert_state_close(pool[slot, h].double().numpy(), ref)


def test_align_commit_bit_equal_to_raw():
    B, width, bs = 8, 6, 4
    wl = W.custom(B=B, H=2, Q=4, lens=[4, 4, 3, 4, 2, 4, 4, 1], S=1 + B + B * width, seed=45,
                  slots=list(range(1, B + 1)))
    table = torch.tensor((1 + B + np.arange(B * width)).reshape(B, width), dtype=torch.int32,
                         device="cuda")
    nc = torch.tensor(np.random.default_rng(2).integers(0, bs * (width - 1), size=B),
                      dtype=torch.int32, device="cuda")
    pools = []
    for fmt in ("raw", "correction"):
        g = DeviceRun(wl, record_format=fmt)
        g.verify()
        api.kda_commit_align(g.A_log, g.g_bias, g.pool, g.cu, g.slots,
                             g.steps[0]["num_accepted"], g.records, table, nc, block_size=bs,
                             record_rows=g.record_rows, error_word=g.err, **g.kw())
        torch.cuda.synchronize()
        assert int(g.err.item()) == 0
        pools.append(g.pool)
    assert torch.equal(pools[0], pools[1])


def test_records_buffer_too_small_is_refused():
    wl = W.custom(B=2, H=1, Q=4, lens=[4, 4], S=4, seed=1)
    g = DeviceRun(wl)                                  # a raw-sized buffer
    with pytest.raises(ValueError):
        api.kda_verify(g.steps[0]["qkv"][:, 0], g.steps[0]["qkv"][:, 1],
                       g.steps[0]["qkv"][:, 2], g.steps[0]["g_raw"],
                       g.steps[0]["beta_buf"][:, :1], g.A_log, g.g_bias, g.pool, g.cu, g.slots,
                       g.records, g.out, window=4, record_slots=wl.spec.record_slots,
                       record_format="correction")


def test_full_size_deferred_two_steps():
    """deferred2 at full size (1024 requests x 16 heads, two steps, the
    benchmark's launch sequence): the correction format gives the raw
    format's final states bit for bit, and a sample of tiles and outputs
    matches the oracle in both formats."""
    wl = W.generate("deferred2")
    sp = wl.spec
    ones = torch.ones(sp.B, dtype=torch.uint8, device="cuda")
    outs, pools = [], []
    for fmt in ("raw", "correction"):
        g = DeviceRun(wl, sentinel=False, record_format=fmt)
        g.verify(0, pending=True)
        g.commit(0, deferred=True)
        g.verify(1, pending=True)
        g.commit(1, deferred=True, eager=ones)
        torch.cuda.synchronize()
        assert int(g.err.item()) == 0
        outs.append(g.out)
        pools.append(g.pool)
        del g
    assert torch.equal(pools[0], pools[1])
    rng = np.random.default_rng(3)
    rows = sorted(rng.choice(sp.B, size=12, replace=False).tolist())
    heads = sorted(rng.choice(sp.H, size=2, replace=False).tolist())
    layer = oracle_layer(wl)
    cache = oracle_cache(wl, "correction")
    s1, s2 = oracle_step(wl, 0), oracle_step(wl, 1)
    O.verify(layer, cache, s1, pending=True, rows=rows, heads=heads)
    O.commit(layer, cache, s1, wl.steps[0].num_accepted.numpy(), deferred=True,
             eager=wl.steps[0].eager.numpy(), rows=rows, heads=heads)
    r2 = O.verify(layer, cache, s2, pending=True, rows=rows, heads=heads)
    O.commit(layer, cache, s2, wl.steps[1].num_accepted.numpy(), rows=rows, heads=heads)
    assert_out_close(outs[1], r2.out)
    assert_out_close(outs[0], r2.out)
    assert cache.written
    for (slot, h), ref in cache.written.items():
        assert_state_close(pools[1][slot, h].double().cpu().numpy(), ref)
