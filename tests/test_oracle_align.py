"""Pins of the oracle's align-mode commit (CPU).

Align mode keeps the recurrent and conv states in paged blocks of
``block_size`` tokens: the state after the last committed token belongs to
the block that holds that token, and a step that completes a block leaves
that block the state at its end.  The pins check the plan by walking the
token positions against explicit block ranges (no division formula), the
replayed states against the oracle verify's own trajectory, the reduction to
the plain commit when every block is the source slot, and the conv windows
against the accepted input sequence.
"""

import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from linear_attention_speculative_kda_gb300 import workloads as W  # noqa: E402
from oracle import kda_oracle as O  # noqa: E402
from tests.helpers import oracle_cache, oracle_layer, oracle_step  # noqa: E402


def _walk(n, num_computed, block_size, width):
    """Final column and (boundary column, boundary_len) by walking positions."""
    blocks = [range(j * block_size, (j + 1) * block_size) for j in range(width + 4)]
    last = num_computed + n - 1
    final_col = next(j for j, blk in enumerate(blocks) if last in blk)
    final_col = min(final_col, width - 1)
    boundary = None
    for t in range(n):
        done = num_computed + t + 1          # tokens in the sequence after token t
        for j, blk in enumerate(blocks):
            if done == blk[-1] + 1 and blk[-1] >= num_computed:
                boundary = (j, t + 1)
                break
        if boundary:
            break
    return final_col, boundary


@pytest.mark.parametrize("block_size", [4, 5, 8, 16])
def test_plan_matches_walk_over_positions(block_size):
    width = 6
    row = [100 + j for j in range(width)]
    for num_computed in range(0, block_size * width - 1):
        for n in range(1, min(block_size, 8) + 1):
            plan = O.align_plan(n, num_computed, row, block_size)
            final_col, boundary = _walk(n, num_computed, block_size, width)
            if boundary is not None and boundary[0] >= width:
                assert plan is None
                continue
            assert plan.final == row[final_col]
            if boundary is None:
                assert plan.boundary == 0
            else:
                assert (plan.boundary, plan.boundary_len) == (row[boundary[0]], boundary[1])


def _align_case(seed=21, Q=4, bs=4):
    wl = W.custom(B=8, H=2, Q=Q, lens=[4, 4, 3, 4, 2, 4, 4, 1], S=60, seed=seed,
                  slots=[1, 2, 3, 0, 4, 5, 6, 7])
    rng = np.random.default_rng(seed)
    width = 6
    # distinct block slots 10.. per row
    table = np.arange(10, 10 + 8 * width).reshape(8, width)
    num_computed = rng.integers(0, bs * (width - 1), size=8)
    return wl, table, num_computed, bs


def test_states_are_the_verify_trajectory_at_final_and_boundary():
    wl, table, nc, bs = _align_case()
    layer, step = oracle_layer(wl), oracle_step(wl)
    ref = O.verify(layer, oracle_cache(wl), step, want_traj=True)
    cache = oracle_cache(wl)
    O.verify(layer, cache, step)                       # writes the records
    acc = wl.steps[0].num_accepted.numpy()
    issues = O.commit_align(layer, cache, step, acc, table, nc, bs)
    assert issues == []
    cu = wl.cu_seqlens.numpy()
    written = set()
    for b in range(8):
        slot = int(wl.state_indices[b])
        n = O.commit_len(acc[b], cu[b + 1] - cu[b], wl.spec.Q)
        if slot <= 0 or n <= 0:
            continue
        plan = O.align_plan(n, int(nc[b]), table[b], bs)
        for h in range(wl.spec.H):
            assert np.array_equal(cache.state(plan.final, h), ref.traj[(cu[b] + n - 1, h)])
            written.add((plan.final, h))
            if plan.boundary > 0 and plan.boundary_len < n:
                assert np.array_equal(cache.state(plan.boundary, h),
                                      ref.traj[(cu[b] + plan.boundary_len - 1, h)])
                written.add((plan.boundary, h))
    assert set(cache.written) == written               # nothing else, not the sources


def test_blocks_all_at_source_is_the_plain_commit():
    wl, _, nc, bs = _align_case(seed=22)
    table = np.repeat(wl.state_indices.numpy()[:, None], 6, axis=1)
    layer, step = oracle_layer(wl), oracle_step(wl)
    acc = wl.steps[0].num_accepted.numpy()
    a, p = oracle_cache(wl), oracle_cache(wl)
    O.verify(layer, a, step)
    O.verify(layer, p, step)
    assert O.commit_align(layer, a, step, acc, table, nc, bs) == []
    assert O.commit(layer, p, step, acc) == []
    assert set(a.written) == set(p.written)
    for key in p.written:
        assert np.array_equal(a.written[key], p.written[key])


def test_conv_windows_follow_the_accepted_sequence():
    rng = np.random.default_rng(30)
    Q, hist, bs, width_bt = 4, 3, 4, 5
    B, S, C = 6, 60, 3
    slots = np.arange(1, B + 1)
    table = np.arange(20, 20 + B * width_bt).reshape(B, width_bt)
    nc = rng.integers(0, bs * (width_bt - 1), size=B)
    acc = rng.integers(1, Q + 1, size=B)
    cu = np.arange(0, Q * (B + 1), Q)
    pool = rng.integers(-10**6, 10**6, size=(S, C, hist + Q - 1)).astype(np.int64)
    seqs = {}
    for s in slots:
        hst = rng.integers(0, 10**6, size=(C, hist))
        x = rng.integers(0, 10**6, size=(C, Q))
        pool[s] = np.concatenate([hst[:, 1:], x], axis=1)
        seqs[int(s)] = (hst, x)
    out, issues = O.conv_compact_align(pool, cu, slots, acc, Q, table, nc, bs)
    assert issues == []
    for b, s in enumerate(slots):
        hst, x = seqs[int(s)]
        n = int(acc[b])
        plan = O.align_plan(n, int(nc[b]), table[b], bs)
        for c in range(C):
            seq = list(hst[c]) + list(x[c])
            assert list(out[plan.final, c, :hist]) == seq[:hist + n][-hist:]
            if plan.boundary > 0 and plan.boundary != plan.final:
                assert list(out[plan.boundary, c, :hist]) == seq[:hist + plan.boundary_len][-hist:]
        # the source slot keeps its post-verify layout (it is neither block)
        assert np.array_equal(out[s], pool[s])


def test_conv_align_with_blocks_at_source_is_the_plain_compaction():
    rng = np.random.default_rng(31)
    Q, B, S = 4, 7, 12
    pool = rng.normal(size=(S, 5, 6))
    slots = np.array([1, 2, 0, 4, 5, 6, 7])
    cu = np.concatenate([[0], np.cumsum(rng.integers(0, Q + 1, size=B))])
    acc = rng.integers(-1, Q + 2, size=B)
    table = np.repeat(slots[:, None], 4, axis=1)
    nc = rng.integers(0, 12, size=B)
    a, ia = O.conv_compact_align(pool, cu, slots, acc, Q, table, nc, 4)
    p, ip = O.conv_compact(pool, cu, slots, acc, Q)
    assert ia == ip == []
    assert np.array_equal(a, p)


def test_invalid_blocks_are_reported():
    wl, table, nc, bs = _align_case(seed=23)
    layer, step = oracle_layer(wl), oracle_step(wl)
    cache = oracle_cache(wl)
    O.verify(layer, cache, step)
    acc = np.full(8, 2)
    table = table.copy()
    table[0, :] = 999                          # final block beyond the pool
    nc = nc.copy()
    nc[1] = bs * 6 + bs - 1                    # boundary block beyond the table
    issues = O.commit_align(layer, cache, step, acc, table, nc, bs)
    assert [(i.row, i.reason) for i in issues][:2] == [(0, "slot"), (1, "block")]


def _deferred_case():
    """Six rows whose state slot is the block of their last computed token
    (column (c - 1) // bs of their table row, as a runner keeps it): row 0
    stays in that block, row 1 starts the next block, row 2 crosses a
    boundary before its last token, row 3 is eager, row 4 accepts nothing,
    row 5 reaches the boundary exactly at its last token."""
    wl = W.custom(B=6, H=2, Q=4, lens=[4] * 6, S=60, seed=33, slots=[1, 2, 3, 4, 5, 6])
    bs, width = 8, 4
    nc = np.array([10, 16, 13, 10, 10, 12])
    table = np.arange(20, 20 + 6 * width).reshape(6, width)
    for b in range(6):
        table[b, (nc[b] - 1) // bs] = int(wl.state_indices[b])
    acc = np.array([3, 4, 4, 2, 0, 4])
    eager = np.array([0, 0, 0, 1, 0, 0], np.uint8)
    return wl, table, nc, bs, acc, eager


def test_deferred_align_commits_only_rows_that_leave_their_block():
    wl, table, nc, bs, acc, eager = _deferred_case()
    layer, step = oracle_layer(wl), oracle_step(wl)
    cache = oracle_cache(wl)
    O.verify(layer, cache, step)
    cache.pending[:] = 7                              # stale counts
    cache.written.clear()
    assert O.commit_align(layer, cache, step, acc, table, nc, bs, deferred=True,
                          eager=eager) == []
    # rows 0 and 5 keep their state in their own slot: pending replays
    assert cache.pending.tolist() == [3, 0, 0, 0, 0, 4]
    # rows 1, 2 (final and boundary block) and 3 are committed now
    final = {b: O.align_plan(int(acc[b]), int(nc[b]), table[b], bs) for b in (1, 2, 3)}
    want = {(final[b].final, h) for b in (1, 2, 3) for h in range(2)}
    want |= {(final[2].boundary, h) for h in range(2)}
    assert final[2].boundary_len == 3 and final[3].final == int(wl.state_indices[3])
    assert set(cache.written) == want


def test_deferred_align_then_flush_equals_the_eager_align_commit():
    wl, table, nc, bs, acc, eager = _deferred_case()
    layer, step = oracle_layer(wl), oracle_step(wl)
    eager_cache, deferred_cache = oracle_cache(wl), oracle_cache(wl)
    for c in (eager_cache, deferred_cache):
        O.verify(layer, c, step)
    assert O.commit_align(layer, eager_cache, step, acc, table, nc, bs) == []
    assert O.commit_align(layer, deferred_cache, step, acc, table, nc, bs, deferred=True,
                          eager=eager) == []
    assert O.flush(layer, deferred_cache, step) == []
    for s in range(wl.spec.S):
        for h in range(wl.spec.H):
            assert np.array_equal(eager_cache.state(s, h), deferred_cache.state(s, h)), (s, h)


# --- record_state_blocks: the running state column after an align commit ---

def _column_of(position, block_size, width):
    """Block-table column holding a token position, by walking the block
    ranges (no division), the last column when it runs past the table."""
    j = 0
    while position >= (j + 1) * block_size:
        j += 1
    return min(j, width - 1)


def test_record_state_blocks_column_by_walk():
    rng = np.random.default_rng(11)
    R, S, bs, width = 40, 50, 16, 6
    idx = rng.permutation(S)[:R].astype(np.int64)
    idx[rng.random(R) < 0.2] = -1                       # requests without a running slot
    nc = rng.integers(0, 120, size=R)
    ns = rng.integers(0, 9, size=R)
    col0 = rng.integers(0, 99, size=S)
    acc0 = rng.integers(2, 9, size=S)
    col, acc, issues = O.record_state_blocks(idx, ns, nc, col0, acc0, bs, width)
    assert issues == []
    touched = set()
    for q in range(R):
        s = int(idx[q])
        if s < 0:
            continue
        touched.add(s)
        assert col[s] == _column_of(max(nc[q] + ns[q] - 1, 0), bs, width)
        assert acc[s] == 1
    for s in range(S):
        if s not in touched:
            assert col[s] == col0[s] and acc[s] == acc0[s]


def test_record_state_blocks_points_at_the_commit_final_block():
    """With the sampled count equal to the commit count n, the recorded
    column holds the block the align commit wrote the final state to."""
    rng = np.random.default_rng(12)
    bs, width, R = 8, 5, 60
    table = np.arange(1, R * width + 1).reshape(R, width)   # distinct block ids
    nc = rng.integers(0, 45, size=R)
    n = rng.integers(1, 9, size=R)
    idx = np.arange(R)
    col, _, issues = O.record_state_blocks(idx, n, nc, np.zeros(R, np.int64),
                                           np.zeros(R, np.int64), bs, width)
    assert issues == []
    for q in range(R):
        plan = O.align_plan(int(n[q]), int(nc[q]), table[q], bs)
        if plan is None:       # the boundary block lies past the table
            continue
        assert table[q][col[q]] == plan.final


def test_record_state_blocks_hand_cases():
    # block_size 16, width 4; per request (slot, num_computed, num_sampled):
    #   q0: slot 2, 30 + 3 - 1 = 32  -> column 2
    #   q1: slot -1                   -> nothing
    #   q2: slot 0, max(0 + 0 - 1, 0) = 0 -> column 0
    #   q3: slot 5, 60 + 10 - 1 = 69 -> column 4, clamped to 3
    #   q4: slot 3, 15 + 1 - 1 = 15  -> column 0 (last position of block 0)
    #   q5: slot 4, 16 + 1 - 1 = 16  -> column 1 (first position of block 1)
    idx = [2, -1, 0, 5, 3, 4]
    nc = [30, 7, 0, 60, 15, 16]
    ns = [3, 2, 0, 10, 1, 1]
    col, acc, issues = O.record_state_blocks(idx, ns, nc, [9] * 6, [7] * 6, 16, 4)
    assert issues == []
    assert col.tolist() == [0, 9, 2, 0, 1, 3]
    assert acc.tolist() == [1, 7, 1, 1, 1, 1]
    # spec rows through request_indices: only requests 3 and 0
    col, acc, _ = O.record_state_blocks(idx, ns, nc, [9] * 6, [7] * 6, 16, 4,
                                        request_indices=[3, 0])
    assert col.tolist() == [9, 9, 2, 9, 9, 3]
    assert acc.tolist() == [7, 7, 1, 7, 7, 1]


def test_record_state_blocks_skips_and_reports():
    idx = [0, 7, 1]          # request 1's slot 7 is past the 4 running slots
    col, acc, issues = O.record_state_blocks(idx, [1, 1, 1], [0, 0, 40], [5] * 4, [5] * 4, 16, 8,
                                             request_indices=[0, 3, 1, 2])
    # row 1 names request 3 (outside the 3 requests): "block"; row 2 -> request
    # 1 -> slot 7: "slot"; rows 0 and 3 record columns 0 and 2
    assert [(i.row, i.reason) for i in issues] == [(1, "block"), (2, "slot")]
    assert col.tolist() == [0, 2, 5, 5]
    assert acc.tolist() == [1, 1, 5, 5]
