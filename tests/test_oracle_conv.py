"""Pins of the oracle's conv-state compaction (CPU).

The compaction of recoverssm.py (``_compact_conv_state_kernel``) rests on one
fact about the short causal conv: after the verify, a row's conv state holds
``[history[1:], x_0 .. x_{Q-1}]``, and once n tokens are accepted the next
step needs, at columns 0 .. history-1, the last ``history`` inputs of the
accepted sequence ``history, x_0 .. x_{n-1}``.  The tests build conv states
from known sequences and check that fact by list slicing, independently of
the oracle's column arithmetic, plus a hand-worked case and the cases the
kernel skips.
"""

import json
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from oracle import kda_oracle as O  # noqa: E402

GOLDEN = os.path.join(ROOT, "tests", "golden", "conv_compact.json")


def _pool_from_sequences(rng, S, C, hist, Q, rows):
    """A pool [S, C, hist + Q - 1] whose row slots hold the post-verify
    layout of known sequences; returns the pool and, per slot, the
    (history, drafts) pair of every channel."""
    width = hist + Q - 1
    pool = rng.integers(-10**6, 10**6, size=(S, C, width)).astype(np.int64)
    seqs = {}
    for slot in rows:
        hst = rng.integers(0, 10**6, size=(C, hist))
        x = rng.integers(0, 10**6, size=(C, Q))
        pool[slot] = np.concatenate([hst[:, 1:], x], axis=1)
        seqs[slot] = (hst, x)
    return pool, seqs


@pytest.mark.parametrize("Q,hist", [(1, 1), (1, 3), (2, 3), (4, 3), (8, 3), (4, 1), (8, 5), (3, 7)])
def test_window_is_last_history_of_accepted_sequence(Q, hist):
    rng = np.random.default_rng(100 * Q + hist)
    S, C, B = 12, 5, 9
    slots = rng.permutation(np.arange(1, S))[:B]
    pool, seqs = _pool_from_sequences(rng, S, C, hist, Q, slots)
    lens = np.full(B, Q)
    cu = np.concatenate([[0], np.cumsum(lens)])
    acc = rng.integers(0, Q + 1, size=B)
    out, issues = O.conv_compact(pool, cu, slots, acc, Q)
    assert issues == []
    for b, slot in enumerate(slots):
        hst, x = seqs[slot]
        n = int(acc[b])
        if n == 0:
            assert np.array_equal(out[slot], pool[slot])
            continue
        for c in range(C):
            accepted = list(hst[c]) + list(x[c, :n])
            assert list(out[slot, c, :hist]) == accepted[-hist:]
        # columns from `hist` on are left as they were
        assert np.array_equal(out[slot, :, hist:], pool[slot, :, hist:])
    untouched = sorted(set(range(S)) - set(int(s) for s in slots))
    assert np.array_equal(out[untouched], pool[untouched])


def test_hand_worked_case():
    g = json.load(open(GOLDEN))
    pool = np.array(g["pool"], dtype=np.int64)
    out, issues = O.conv_compact(pool, g["cu_seqlens"], g["state_indices"],
                                 g["num_accepted"], g["window"])
    assert issues == []
    assert out.tolist() == g["expected"]


def test_one_accepted_token_is_identity():
    rng = np.random.default_rng(3)
    pool = rng.normal(size=(4, 6, 7))
    out, _ = O.conv_compact(pool, [0, 4, 8], [1, 3], [1, 1], 4)
    assert np.array_equal(out, pool)


def test_skipped_rows_and_clamps():
    rng = np.random.default_rng(4)
    Q, hist = 4, 3
    pool = rng.normal(size=(6, 3, hist + Q - 1))
    cu = [0, 4, 8, 8, 10, 14, 18]
    slots = [1, 0, 2, 3, 4, 5]
    # rows: n = 0; null slot; T == 0; 99 clamped to T = 2; -5 clamped to 0; n = 2
    acc = [0, 3, 3, 99, -5, 2]
    out, issues = O.conv_compact(pool, cu, slots, acc, Q)
    assert issues == []
    for s in (0, 1, 2, 4):
        assert np.array_equal(out[s], pool[s])
    for s in (3, 5):  # n = 2: the window starting at column 1
        assert np.array_equal(out[s, :, :hist], pool[s, :, 1:1 + hist])
        assert np.array_equal(out[s, :, hist:], pool[s, :, hist:])


def test_invalid_rows_are_reported_and_skipped():
    rng = np.random.default_rng(5)
    pool = rng.normal(size=(4, 2, 5))
    out, issues = O.conv_compact(pool, [0, 4, 9, 12], [1, 2, 7], [2, 2, 2], 3)
    assert [(i.row, i.reason) for i in issues] == [(0, "length"), (1, "length"), (2, "slot")]
    assert np.array_equal(out, pool)


def test_history_of_width_and_window():
    assert O.conv_history(6, 4) == 3
    assert O.conv_history(3, 1) == 3
    with pytest.raises(ValueError):
        O.conv_compact(np.zeros((2, 1, 2)), [0, 1], [1], [1], 4)
