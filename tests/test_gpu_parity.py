"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Tolerances (from the method's target, written here as the tests apply them):
- bf16 outputs: |gpu - oracle| <= 2e-3 element by element, the oracle value
  unrounded (double precision), and within half a bf16 ulp of the oracle
  value plus 1e-7 (the rounding bound, helpers.assert_out_close);
- fp32 states: normwise per (slot, head) tile, max |gpu - oracle| <=
  1e-5 * max |oracle|;
- commit vs the verify trajectory on the GPU: bit-identical;
- records: bit-identical copies of the raw bf16 inputs.
"""

import numpy as np
import pytest
import torch

from linear_attention_speculative_kda_gb300 import api
from linear_attention_speculative_kda_gb300 import workloads as W
from oracle import kda_oracle as O
from tests.helpers import (DeviceRun, assert_out_close, assert_state_close, f64, oracle_cache,
                           oracle_layer, oracle_step)

pytestmark = pytest.mark.gpu

REC = api.RECORD_STRIDE


def _small_cases():
    # several tiles, ragged tails (T < Q), an empty row, null rows, both gates
    yield "ragged_q8", W.custom(B=12, H=3, Q=8, lens=[8, 1, 5, 0, 8, 3, 7, 2, 8, 6, 4, 8],
                                S=16, seed=1)
    yield "bounded_q8", W.custom(B=10, H=2, Q=8, lens=[8, 8, 2, 7, 5, 8, 1, 3, 8, 6], S=13,
                                 bounded=True, lower_bound=-5.0, seed=2,
                                 slots=[3, 0, 5, 7, 0, 1, 9, 11, 2, 12])
    yield "q1", W.custom(B=6, H=4, Q=1, lens=[1, 1, 0, 1, 1, 1], S=8, seed=3)
    yield "tiny", W.generate("tiny")


@pytest.mark.parametrize("name,wl", list(_small_cases()), ids=lambda x: x if isinstance(x, str) else "")
def test_verify_outputs_records_trajectory(name, wl):
    g = DeviceRun(wl, with_traj=True)
    g.verify()
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    layer, step = oracle_layer(wl), oracle_step(wl)
    cache = oracle_cache(wl)
    res = O.verify(layer, cache, step, want_traj=True)
    assert_out_close(g.out, res.out)
    # skipped rows keep the sentinel output
    cu = wl.cu_seqlens.numpy()
    run = set(res.rows_run)
    out = f64(g.out)
    for b in range(wl.spec.B):
        if b not in run:
            assert (out[cu[b]:cu[b + 1]] == -9.0).all()
    # the pool is not written by a verify without pending
    assert torch.equal(g.pool, g.pool0)
    # trajectory: every token's state within tolerance
    traj = g.traj.cpu().numpy()
    for (tok, h), ref in res.traj.items():
        assert_state_close(traj[tok, h].astype(np.float64), ref)
    # records are the raw inputs, bit for bit
    sp = wl.spec
    rec = g.records.view(torch.int16).cpu().reshape(sp.record_slots + 1, sp.H, sp.Q, REC)
    st = wl.steps[0]
    for b in run:
        bos, T = cu[b], cu[b + 1] - cu[b]
        r = b if wl.record_rows is None else int(wl.record_rows[b])
        for h in range(sp.H):
            got = rec[r + 1, h, :T]
            assert torch.equal(got[:, :128], st.k[bos:bos + T, h].view(torch.int16))
            assert torch.equal(got[:, 128:256], st.v[bos:bos + T, h].view(torch.int16))
            assert torch.equal(got[:, 256:384], st.g_raw[bos:bos + T, h].view(torch.int16))
            assert torch.equal(got[:, 384], st.beta_raw[bos:bos + T, h].view(torch.int16))


@pytest.mark.parametrize("name,wl", list(_small_cases()), ids=lambda x: x if isinstance(x, str) else "")
def test_commit_matches_oracle_and_trajectory_bits(name, wl):
    g = DeviceRun(wl, with_traj=True)
    g.verify()
    g.commit()
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    layer, step = oracle_layer(wl), oracle_step(wl)
    cache = oracle_cache(wl)
    O.verify(layer, cache, step)
    acc = wl.steps[0].num_accepted.numpy()
    O.commit(layer, cache, step, acc)
    pool = g.pool.cpu()
    pool0 = g.pool0.cpu()
    written = {s for (s, _) in cache.written}
    cu = wl.cu_seqlens.numpy()
    for b in range(wl.spec.B):
        slot = int(wl.state_indices[b])
        T = cu[b + 1] - cu[b]
        n = O.commit_len(acc[b], T, wl.spec.Q)
        for h in range(wl.spec.H):
            if slot in written:
                assert_state_close(pool[slot, h].double().numpy(), cache.written[(slot, h)])
                # bit-exact against the verify's own state after token n
                assert torch.equal(pool[slot, h], g.traj[cu[b] + n - 1, h].cpu())
            elif slot > 0:
                assert torch.equal(pool[slot, h], pool0[slot, h])
    # slots no row owns are untouched
    owned = set(int(s) for s in wl.state_indices)
    for s in range(wl.spec.S):
        if s not in owned:
            assert torch.equal(pool[s], pool0[s])


def test_deferred_two_steps_bit_exact_and_oracle():
    wl = W.custom(B=16, H=2, Q=4, lens=[4] * 13 + [2, 3, 1], S=20, R=24, deferred=True,
                  steps=2, seed=7, eager_prob=0.25)
    acc1 = wl.steps[0].num_accepted
    acc2 = wl.steps[1].num_accepted
    # eager two steps on the GPU
    ge = DeviceRun(wl)
    ge.verify(0)
    ge.commit(0)
    oe1 = ge.out.clone()
    ge.verify(1)
    ge.commit(1)
    # deferred: verify1, deferred commit1, fused verify2, eager commit2
    gd = DeviceRun(wl)
    gd.verify(0, pending=True)
    gd.commit(0, deferred=True)
    od1 = gd.out.clone()
    pend = gd.pending.clone()
    gd.verify(1, pending=True)
    gd.commit(1, deferred=True, eager=torch.ones_like(wl.steps[1].eager).cuda())
    torch.cuda.synchronize()
    assert int(ge.err.item()) == 0 and int(gd.err.item()) == 0
    assert torch.equal(oe1, od1)
    assert torch.equal(ge.out, gd.out)
    assert torch.equal(ge.pool, gd.pool)
    assert int(gd.pending.abs().sum()) == 0
    # pending after step 1 is what the plan says
    rr = wl.record_rows.numpy()
    cu = wl.cu_seqlens.numpy()
    eg = wl.steps[0].eager.numpy()
    exp_p = np.zeros(wl.spec.record_slots, np.int64)
    for b in range(wl.spec.B):
        n = O.commit_len(int(acc1[b]), cu[b + 1] - cu[b], wl.spec.Q)
        valid = int(wl.state_indices[b]) > 0 and n > 0
        exp_p[rr[b]] = n if (valid and not eg[b]) else 0
    assert pend.cpu().numpy().tolist() == exp_p.tolist()
    # and both match the oracle's two steps
    layer = oracle_layer(wl)
    cache = oracle_cache(wl)
    s1, s2 = oracle_step(wl, 0), oracle_step(wl, 1)
    O.verify(layer, cache, s1, pending=True)
    O.commit(layer, cache, s1, acc1.numpy(), deferred=True, eager=eg)
    r2 = O.verify(layer, cache, s2, pending=True)
    O.commit(layer, cache, s2, acc2.numpy())
    assert_out_close(gd.out, r2.out)
    pool = gd.pool.cpu()
    for (slot, h), ref in cache.written.items():
        assert_state_close(pool[slot, h].double().numpy(), ref)


def test_flush_then_plain_verify_equals_fused_verify():
    wl = W.custom(B=8, H=2, Q=4, lens=[4, 4, 3, 4, 2, 4, 4, 1], S=12, R=10, deferred=True,
                  steps=2, seed=9)
    ga = DeviceRun(wl)
    ga.verify(0, pending=True)
    ga.commit(0, deferred=True)
    ga.verify(1, pending=True)
    gb = DeviceRun(wl)
    gb.verify(0, pending=True)
    gb.commit(0, deferred=True)
    pend = gb.pending.clone()
    gb.flush()
    assert torch.equal(gb.pending, pend)       # flush leaves pending
    gb.verify(1, pending=False)
    torch.cuda.synchronize()
    assert torch.equal(ga.out, gb.out)
    assert torch.equal(ga.pool, gb.pool)


def test_error_word_and_skips():
    wl = W.custom(B=5, H=2, Q=4, lens=[4, 4, 4, 4, 4], S=8, R=6, seed=13,
                  slots=[1, 2, 3, 4, 5], record_rows=[0, 1, 2, 3, 4])
    g = DeviceRun(wl)
    cu = torch.tensor([0, 4, 9, 12, 16, 20], dtype=torch.int32, device="cuda")   # row 1: T = 5
    slots = torch.tensor([1, 2, 11, 4, 5], dtype=torch.int32, device="cuda")     # row 2: 11 >= S
    rr = torch.tensor([0, 1, 2, 9, 4], dtype=torch.int32, device="cuda")         # row 3: 9 >= R
    g.verify(cu=cu, slots=slots, record_rows=rr)
    torch.cuda.synchronize()
    assert int(g.err.item()) == api.ROW_BAD_LENGTH | api.ROW_BAD_SLOT | api.ROW_BAD_RECORD
    out = f64(g.out)
    assert (out[4:16] == -9.0).all()           # rows 1..3 skipped
    assert not (out[0:4] == -9.0).any()        # rows 0 and 4 ran
    assert not (out[16:20] == -9.0).any()
    g.err.zero_()
    g.pending[0] = 7                            # > Q
    g.verify(cu=cu, slots=slots, record_rows=rr, pending=True)
    torch.cuda.synchronize()
    assert int(g.err.item()) & api.ROW_BAD_PENDING
    assert torch.equal(g.pool, g.pool0)


def test_zero_rows_and_host_errors():
    wl = W.custom(B=2, H=1, Q=4, lens=[4, 4], S=4, seed=1)
    g = DeviceRun(wl)
    empty = torch.zeros(0, dtype=torch.int32, device="cuda")
    st = g.steps[0]
    api.kda_verify(st["qkv"][:, 0], st["qkv"][:, 1], st["qkv"][:, 2], st["g_raw"],
                   st["beta_buf"][:, :1], g.A_log, g.g_bias, g.pool,
                   torch.zeros(1, dtype=torch.int32, device="cuda"), empty, g.records, g.out,
                   window=4, record_slots=2)
    with pytest.raises(api.KDAError) as ei:
        api.kda_verify(st["qkv"][:, 0], st["qkv"][:, 1], st["qkv"][:, 2], st["g_raw"],
                       st["beta_buf"][:, :1], g.A_log, g.g_bias, g.pool, g.cu, g.slots,
                       g.records, g.out, window=9, record_slots=2)
    assert ei.value.status == api.KDA_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.equal(g.pool, g.pool0)


@pytest.mark.parametrize("name", ["mtp3", "dflash7", "mixed", "deferred2"])
def test_full_size_sampled(name):
    """Full-size workloads in the benchmark's launch configuration: every
    commit is bit-checked against the verify trajectory on the GPU, and a
    sample of (row, head) tiles is checked against the oracle."""
    wl = W.generate(name)
    sp = wl.spec
    g = DeviceRun(wl, with_traj=True, sentinel=False)
    deferred = sp.deferred
    g.verify(0, pending=deferred)
    g.commit(0, deferred=deferred)
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    rng = np.random.default_rng(0)
    rows = sorted(rng.choice(sp.B, size=min(sp.B, 24), replace=False).tolist())
    heads = sorted(rng.choice(sp.H, size=min(sp.H, 3), replace=False).tolist())
    layer, step = oracle_layer(wl), oracle_step(wl)
    cache = oracle_cache(wl)
    res = O.verify(layer, cache, step, pending=deferred, rows=rows, heads=heads)
    acc = wl.steps[0].num_accepted.numpy()
    eager = None if wl.steps[0].eager is None else wl.steps[0].eager.numpy()
    O.commit(layer, cache, step, acc, deferred=deferred, eager=eager, rows=rows, heads=heads)
    assert_out_close(g.out, res.out)
    pool = g.pool
    for (slot, h), ref in cache.written.items():
        assert_state_close(pool[slot, h].double().cpu().numpy(), ref)
    # every committed tile equals the verify trajectory bits (all rows and heads)
    cu = wl.cu_seqlens.numpy()
    slots = wl.state_indices.numpy()
    committed, toks = [], []
    for b in range(sp.B):
        n = O.commit_len(int(acc[b]), cu[b + 1] - cu[b], sp.Q)
        now = eager is None or bool(eager[b])
        if slots[b] > 0 and n > 0 and (not deferred or now):
            committed.append(int(slots[b]))
            toks.append(int(cu[b]) + n - 1)
    if committed:
        idx_s = torch.tensor(committed, device="cuda")
        idx_t = torch.tensor(toks, device="cuda")
        assert torch.equal(pool[idx_s], g.traj[idx_t])
    if deferred:
        # pending rows were not written
        rr = wl.record_rows.numpy()
        p = g.pending.cpu().numpy()
        for b in range(sp.B):
            if p[rr[b]] > 0:
                assert torch.equal(pool[int(slots[b])], g.pool0[int(slots[b])])


def test_all_rows_idle_and_more_ctas_than_work():
    # every row null or empty: the persistent CTAs find no work and write nothing
    wl = W.custom(B=40, H=16, Q=4, lens=[0, 4] * 20, S=48, seed=17,
                  slots=[0 if i % 2 else i + 1 for i in range(40)])
    g = DeviceRun(wl)
    g.verify()
    g.commit()
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    assert torch.equal(g.pool, g.pool0)
    assert (f64(g.out) == -9.0).all()


def test_strided_activations_eight_byte_aligned():
    """Activation rows whose token stride is a multiple of 4 elements but not of
    8, starting 8 bytes past a 16-byte boundary, give the same bits as the
    packed layout."""
    wl = W.custom(B=9, H=3, Q=8, lens=[8, 3, 0, 8, 5, 1, 8, 7, 2], S=12, seed=23)
    ref = DeviceRun(wl, with_traj=True)
    ref.verify()
    ref.commit()
    g = DeviceRun(wl, with_traj=True)
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
                   g.slots, g.records, g.out, trajectory_out=g.traj, error_word=g.err, **g.kw())
    g.commit()
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0 and int(ref.err.item()) == 0
    assert torch.equal(g.out, ref.out)
    assert torch.equal(g.traj, ref.traj)
    assert torch.equal(g.pool, ref.pool)
    assert torch.equal(g.records, ref.records)


def test_deferred_window8_bounded_with_folds():
    """Window 8 with the bounded gate and pending folds (token-vector buffers
    sized for 16 tokens): two deferred steps equal two eager steps bit for
    bit and match the oracle."""
    wl = W.custom(B=24, H=2, Q=8, lens=[8, 7, 1, 8, 3, 8, 8, 5, 0, 8, 2, 8] * 2, S=30, R=28,
                  deferred=True, steps=2, seed=29, bounded=True, lower_bound=-5.0,
                  eager_prob=0.2)
    ge = DeviceRun(wl)
    ge.verify(0)
    ge.commit(0)
    ge.verify(1)
    ge.commit(1)
    gd = DeviceRun(wl)
    gd.verify(0, pending=True)
    gd.commit(0, deferred=True)
    gd.verify(1, pending=True)
    gd.commit(1, deferred=True, eager=torch.ones_like(wl.steps[1].eager).cuda())
    torch.cuda.synchronize()
    assert int(ge.err.item()) == 0 and int(gd.err.item()) == 0
    assert torch.equal(ge.out, gd.out)
    assert torch.equal(ge.pool, gd.pool)
    layer = oracle_layer(wl)
    cache = oracle_cache(wl)
    s1, s2 = oracle_step(wl, 0), oracle_step(wl, 1)
    O.verify(layer, cache, s1, pending=True)
    O.commit(layer, cache, s1, wl.steps[0].num_accepted.numpy(), deferred=True,
             eager=wl.steps[0].eager.numpy())
    r2 = O.verify(layer, cache, s2, pending=True)
    O.commit(layer, cache, s2, wl.steps[1].num_accepted.numpy())
    assert_out_close(gd.out, r2.out)
    pool = gd.pool.cpu()
    for (slot, h), ref in cache.written.items():
        assert_state_close(pool[slot, h].double().numpy(), ref)


def test_record_slot_minus_one_rows():
    """Rows without a record slot (-1) verify normally into the scratch row,
    are never committed, and leave pending alone."""
    wl = W.custom(B=6, H=2, Q=4, lens=[4, 4, 4, 4, 4, 4], S=10, R=6, deferred=True, seed=31,
                  record_rows=[0, -1, 2, -1, 4, 5])
    g = DeviceRun(wl)
    g.pending.fill_(0)
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


def test_deferred_commit_clears_pending_of_skipped_rows():
    """A deferred commit that skips rows for bad metadata still rewrites
    their pending counts (to 0) when the record slot is usable, as the
    oracle does; a row with a bad record slot leaves pending alone."""
    wl = W.custom(B=4, H=2, Q=4, lens=[4, 4, 4, 4], S=6, R=6, deferred=True,
                  record_rows=[1, 2, 3, 4], slots=[1, 2, 3, 4], seed=9)
    i32 = dict(dtype=torch.int32, device="cuda")
    cu = torch.tensor([0, 4, 9, 12, 16], **i32)        # row 1: T = 5 > Q
    slots = torch.tensor([1, 2, 9, 3], **i32)           # row 2: slot 9 >= S
    rr = torch.tensor([1, 2, 3, 8], **i32)              # row 3: record slot 8 >= R
    acc = torch.tensor([2, 2, 2, 2], **i32)
    g = DeviceRun(wl)
    g.pending.fill_(3)
    g.commit(deferred=True, eager=torch.zeros(4, dtype=torch.uint8, device="cuda"),
             num_accepted=acc, cu=cu, slots=slots, record_rows=rr)
    torch.cuda.synchronize()
    assert int(g.err.item()) == api.ROW_BAD_LENGTH | api.ROW_BAD_SLOT | api.ROW_BAD_RECORD
    layer = oracle_layer(wl)
    step = oracle_step(wl, cu_seqlens=cu.cpu(), state_indices=slots.cpu(),
                       record_rows=rr.cpu().numpy())
    cache = oracle_cache(wl)
    cache.pending[:] = 3
    O.commit(layer, cache, step, acc.cpu().numpy(), deferred=True, eager=np.zeros(4, np.uint8))
    assert g.pending.cpu().tolist() == cache.pending.tolist() == [3, 2, 0, 0, 3, 3]
    assert torch.equal(g.pool, g.pool0)
