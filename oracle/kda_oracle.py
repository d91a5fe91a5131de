"""CPU oracle of KDA speculative verify and commit (test infrastructure only).

ONLY the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  The product path (the CUDA library and
its Python binding) never does, and this module imports nothing from the
product package.

The arithmetic of one window lives in ``kda_window.c`` (double precision,
the plain definition of the recurrence).  This module adds the bookkeeping
the pages define around it, each function citing the passage it follows:

* ``verify`` -- the RecoverSSM verify of recoverssm.py (``_verify_kernel``):
  per (request row, head), read the checkpoint of ``state_indices[b]``, run
  the row's tokens, write the outputs and record each token's raw k, v,
  g_raw and beta_raw; never store a state.  Rows whose state index is
  <= 0 (the null block) or whose token count is 0 are skipped.  With
  ``pending`` (the deferred commit of the Kimi-K3 page, context.py), the
  pending replay of the row's record slot is folded in first: the recorded
  tokens are replayed from the checkpoint, the folded state is written back
  to the pool, and the new tokens run from it.
* ``commit`` -- ``_prepare_commit_plan_kernel`` plus the replay in
  ``Glm5NextRecoverSSMCommitContext.commit``: n = min(max(accepted, 0), T, Q),
  valid iff the state index is above the null block and n > 0; a valid row's
  checkpoint becomes the state after its first n recorded tokens.  With
  ``pending`` (``KDADeferredCommitContext.commit``): rows not in ``eager``
  only store n as the pending replay of their record slot.
* ``flush`` -- ``KDADeferredCommitContext.flush``: fold pending replays into
  the checkpoints in place, leaving ``pending`` as it is.
* ``commit_align`` / ``conv_compact_align`` -- the align mode of the same
  commit (``_prepare_commit_plan_kernel`` with a block table,
  ``_replay_indices_kernel``): the state after the n-th accepted token goes
  to the block that holds that token, and, when the step crosses a block
  boundary before its last token, the state at the boundary goes to the
  block that ends there; the conv windows follow the same two blocks.
* ``record_state_blocks`` -- ``_record_state_block_kernel`` of recoverssm.py:
  after an align-mode commit, each committed request's running state column
  points at the block holding its last committed token (the final block of
  ``commit_align`` when its sampled count is the commit count n) and its
  accepted count is reset to 1.
* ``conv_compact`` -- ``_compact_conv_state_kernel`` of recoverssm.py in its
  non-align form: after the verify a row's conv state holds
  ``[history[1:], x_0 .. x_{Q-1}]``; once n tokens are accepted the window
  that starts at column n - 1 is moved to column 0, so that the next step
  reads it as if one token had been accepted.

Readings where the pages are silent (the same list is kept with the design
notes): a row with T > Q, a state index >= the pool size, a record slot
outside [-1, R) or a pending count outside [0, Q] is invalid and skipped;
a record slot of -1 is a scratch row that is written but never replayed;
the fold of a pending replay happens even when the row has no new tokens;
``pending`` is rewritten for every row a deferred commit sees (n for valid
deferred rows, 0 otherwise) and is never written by a verify.

Parity pins: see ``tests/test_oracle_pins.py`` (closed forms, brute force,
invariants).
"""

from __future__ import annotations

import contextlib
import ctypes
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

from . import build as _build

_dbl_p = ctypes.POINTER(ctypes.c_double)

_LIBS = {}
_ARITHMETIC = "fp64"


@contextlib.contextmanager
def arithmetic(kind: str):
    """Within the block, run the window loops in ``kind``: "fp64" (the
    oracle) or "fp32" (a float build of the same C file).  Only the
    benchmark's CPU baseline times the float build; the tests never use it."""
    global _ARITHMETIC
    if kind not in ("fp64", "fp32"):
        raise ValueError("arithmetic must be 'fp64' or 'fp32'")
    prev, _ARITHMETIC = _ARITHMETIC, kind
    try:
        yield
    finally:
        _ARITHMETIC = prev


def _lib():
    lib = _LIBS.get(_ARITHMETIC)
    if lib is None:
        path = _build.library(_ARITHMETIC)
        lib = ctypes.CDLL(path)
        lib.kda_oracle_window.restype = ctypes.c_int
        lib.kda_oracle_window.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int,
            _dbl_p,
            _dbl_p, _dbl_p, _dbl_p,
            _dbl_p, _dbl_p,
            ctypes.c_double, _dbl_p,
            ctypes.c_int, ctypes.c_double, ctypes.c_double,
            _dbl_p, _dbl_p, _dbl_p, _dbl_p,
        ]
        lib.kda_oracle_fold_deltas.restype = ctypes.c_int
        lib.kda_oracle_fold_deltas.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int,
            _dbl_p, _dbl_p, _dbl_p, _dbl_p,
            ctypes.c_double, _dbl_p,
            ctypes.c_int, ctypes.c_double,
            _dbl_p,
        ]
        lib.kda_oracle_gate.restype = ctypes.c_double
        lib.kda_oracle_gate.argtypes = [ctypes.c_double, ctypes.c_double,
                                        ctypes.c_int, ctypes.c_double]
        lib.kda_oracle_round_bf16.restype = ctypes.c_double
        lib.kda_oracle_round_bf16.argtypes = [ctypes.c_double]
        _LIBS[_ARITHMETIC] = lib
    return lib


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(_dbl_p)


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def gate(x: float, a_log: float, bounded: bool, lower_bound: float) -> float:
    """Gate value g of one channel for x = g_raw + g_bias (kda.py)."""
    return _lib().kda_oracle_gate(float(x), float(a_log), int(bool(bounded)),
                                  float(lower_bound))


def round_bf16(x: float) -> float:
    """Nearest bfloat16 value of x (ties to even)."""
    return _lib().kda_oracle_round_bf16(float(x))


def window(h0, k, v, g_raw, beta_raw, a_log, g_bias, *, q=None,
           bounded=False, lower_bound=0.0, scale=1.0, want_out=None,
           want_traj=False):
    """Run one window of T tokens from state ``h0`` (V x K).

    ``k``, ``g_raw``: T x K; ``v``: T x V; ``beta_raw``: T; ``q``: T x K or
    None; ``g_bias``: K.  Returns ``(out, traj, h_final)``: ``out`` T x V
    (None without q), ``traj`` T x V x K (None unless asked), ``h_final``
    V x K.
    """
    out, traj, h_final, _ = window_deltas(
        h0, k, v, g_raw, beta_raw, a_log, g_bias, q=q, bounded=bounded,
        lower_bound=lower_bound, scale=scale, want_out=want_out, want_traj=want_traj,
        want_delta=False)
    return out, traj, h_final


def window_deltas(h0, k, v, g_raw, beta_raw, a_log, g_bias, *, q=None,
                  bounded=False, lower_bound=0.0, scale=1.0, want_out=None,
                  want_traj=False, want_delta=True):
    """``window`` plus each token's delta v' = beta (v - H k^) (T x V, the
    fp32 "correction" the Kimi-K3 deferred context records), as a fourth
    result (None unless asked)."""
    h0 = _f64(h0)
    V, K = h0.shape
    k = _f64(k).reshape(-1, K)
    T = k.shape[0]
    v = _f64(v).reshape(T, V)
    g_raw = _f64(g_raw).reshape(T, K)
    beta_raw = _f64(beta_raw).reshape(T)
    g_bias = _f64(g_bias).reshape(K)
    if q is not None:
        q = _f64(q).reshape(T, K)
    if want_out is None:
        want_out = q is not None
    out = np.empty((T, V), np.float64) if want_out else None
    traj = np.empty((T, V, K), np.float64) if want_traj else None
    h_final = np.empty((V, K), np.float64)
    delta = np.empty((T, V), np.float64) if want_delta else None
    rc = _lib().kda_oracle_window(
        K, V, T, _ptr(h0), _ptr(q), _ptr(k), _ptr(v), _ptr(g_raw),
        _ptr(beta_raw), float(a_log), _ptr(g_bias), int(bool(bounded)),
        float(lower_bound), float(scale), _ptr(out), _ptr(traj), _ptr(h_final),
        _ptr(delta))
    if rc != 0:
        raise ValueError("oracle window: bad sizes")
    return out, traj, h_final, delta


def fold_deltas(h0, k, g_raw, delta, a_log, g_bias, *, bounded=False, lower_bound=0.0):
    """The closed form of n tokens whose deltas are known (the Kimi-K3
    fp32-correction commit): H_n = H_0 diag(P_0) + sum_t d_t (k^_t * P_t)^T,
    P_t the product of the later tokens' decays (see ``kda_window.c``).
    ``k``, ``g_raw``: n x K; ``delta``: n x V; returns H_n (V x K)."""
    h0 = _f64(h0)
    V, K = h0.shape
    k = _f64(k).reshape(-1, K)
    n = k.shape[0]
    g_raw = _f64(g_raw).reshape(n, K)
    delta = _f64(delta).reshape(n, V)
    g_bias = _f64(g_bias).reshape(K)
    h_final = np.empty((V, K), np.float64)
    rc = _lib().kda_oracle_fold_deltas(
        K, V, n, _ptr(h0), _ptr(k), _ptr(g_raw), _ptr(delta), float(a_log), _ptr(g_bias),
        int(bool(bounded)), float(lower_bound), _ptr(h_final))
    if rc != 0:
        raise ValueError("oracle fold: bad sizes")
    return h_final


# ---------------------------------------------------------------------------
# What persists between calls: the state pool, the records and pending.
# ---------------------------------------------------------------------------

@dataclass
class Layer:
    """Gate parameters and sizes of one KDA layer (kda.py: A_log per head,
    dt_bias per channel, the optional lower bound, scale = head_dim**-0.5)."""

    num_heads: int
    head_dim: int
    window: int              # Q = 1 + num_spec
    a_log: np.ndarray        # [H]
    g_bias: np.ndarray       # [H, K]
    bounded: bool
    lower_bound: float
    scale: float


@dataclass
class Step:
    """One step's activations (token-major, float64) and row metadata."""

    q: np.ndarray            # [T_tot, H, K]
    k: np.ndarray            # [T_tot, H, K]
    v: np.ndarray            # [T_tot, H, V]
    g_raw: np.ndarray        # [T_tot, H, K]
    beta_raw: np.ndarray     # [T_tot, H]
    cu_seqlens: np.ndarray   # [B+1]
    state_indices: np.ndarray  # [B]
    record_rows: np.ndarray | None = None  # [B], -1 = scratch row


class Cache:
    """The oracle's copy of the state pool, records and pending counts.

    The pool is read lazily from a float32 array ``[S, H, V, K]`` (never
    modified); states the oracle writes are kept as float64 tiles.
    ``record_format``: "raw" records hold each token's k, v, g_raw and
    beta_raw and are replayed through the recurrence; "correction" records
    hold k, g_raw and the token's delta (Kimi-K3's fp32 corrections) and are
    folded in closed form.
    """

    def __init__(self, pool_f32, record_slots: int, pending=None,
                 record_format: str = "raw"):
        if record_format not in ("raw", "correction"):
            raise ValueError("record_format must be 'raw' or 'correction'")
        self.pool_src = pool_f32
        self.num_slots = pool_f32.shape[0]
        self.record_slots = record_slots
        self.record_format = record_format
        self.written: dict[tuple[int, int], np.ndarray] = {}
        self.records: dict[tuple[int, int], dict] = {}
        if pending is None:
            pending = np.zeros(record_slots, np.int64)
        self.pending = np.array(pending, dtype=np.int64, copy=True)

    def state(self, slot: int, head: int) -> np.ndarray:
        tile = self.written.get((slot, head))
        if tile is not None:
            return tile.copy()
        return np.asarray(self.pool_src[slot, head], dtype=np.float64)

    def set_state(self, slot: int, head: int, tile: np.ndarray) -> None:
        self.written[(slot, head)] = np.array(tile, dtype=np.float64, copy=True)


@dataclass
class RowIssue:
    row: int
    reason: str  # "length", "slot", "record", "pending", "block"


@dataclass
class VerifyResult:
    out: np.ndarray                         # [T_tot, H, V], NaN where not written
    traj: dict = field(default_factory=dict)  # (token, head) -> V x K
    issues: list = field(default_factory=list)
    rows_run: list = field(default_factory=list)


def _row_len(cu, b):
    return int(cu[b + 1]) - int(cu[b])


def _record_slot(record_rows, b):
    return b if record_rows is None else int(record_rows[b])


def _row_checks(layer: Layer, cache: Cache, T: int, slot: int, r: int):
    """Checks of one row's metadata; returns the reason it is invalid or None."""
    if T < 0 or T > layer.window:
        return "length"
    if slot >= cache.num_slots:
        return "slot"
    if r < -1 or r >= cache.record_slots:
        return "record"
    return None


def _replay_records(layer, cache, slot, head, r, n):
    """Replay the first n recorded tokens of record slot r from the
    checkpoint (the commit's replay: q is not needed, so no outputs); with
    correction records, fold their deltas in closed form instead."""
    rec = cache.records[(r, head)]
    h0 = cache.state(slot, head)
    if cache.record_format == "correction":
        return fold_deltas(h0, rec["k"][:n], rec["g"][:n], rec["delta"][:n],
                           layer.a_log[head], layer.g_bias[head], bounded=layer.bounded,
                           lower_bound=layer.lower_bound)
    _, _, h = window(h0, rec["k"][:n], rec["v"][:n], rec["g"][:n],
                     rec["beta"][:n], layer.a_log[head], layer.g_bias[head],
                     bounded=layer.bounded, lower_bound=layer.lower_bound,
                     scale=layer.scale)
    return h


def _map_rows(fn, rows, threads):
    if threads and threads > 1 and len(rows) > 1:
        with ThreadPoolExecutor(max_workers=threads) as pool:
            return list(pool.map(fn, rows))
    return [fn(b) for b in rows]


def verify(layer: Layer, cache: Cache, step: Step, *, pending: bool = False,
           rows=None, heads=None, want_traj: bool = False,
           threads: int = 1) -> VerifyResult:
    """RecoverSSM verify (recoverssm.py ``_verify_kernel``), optionally
    folding pending replays first (context.py: the next verify replays the
    pending count of the row's record slot in the same pass).  With
    correction records (``cache.record_format``) each token's record holds
    its k, g_raw and delta instead of k, v, g_raw and beta_raw."""
    B = len(step.state_indices)
    H, D = layer.num_heads, layer.head_dim
    T_tot = step.k.shape[0]
    res = VerifyResult(out=np.full((T_tot, H, D), np.nan))
    rows = range(B) if rows is None else rows
    heads = range(H) if heads is None else heads

    def run(b):
        T = _row_len(step.cu_seqlens, b)
        slot = int(step.state_indices[b])
        r = _record_slot(step.record_rows, b)
        bad = _row_checks(layer, cache, T, slot, r)
        if bad:
            return RowIssue(b, bad)
        if slot <= 0:          # null block: the row is padding
            return None
        p = int(cache.pending[r]) if (pending and r >= 0) else 0
        if p < 0 or p > layer.window:
            return RowIssue(b, "pending")
        if T == 0 and p == 0:
            return None
        bos = int(step.cu_seqlens[b])
        for h in heads:
            if p > 0:
                cache.set_state(slot, h, _replay_records(layer, cache, slot, h, r, p))
            if T == 0:
                continue
            sl = slice(bos, bos + T)
            out, traj, _, delta = window_deltas(
                cache.state(slot, h), step.k[sl, h], step.v[sl, h],
                step.g_raw[sl, h], step.beta_raw[sl, h], layer.a_log[h],
                layer.g_bias[h], q=step.q[sl, h], bounded=layer.bounded,
                lower_bound=layer.lower_bound, scale=layer.scale,
                want_traj=want_traj, want_delta=cache.record_format == "correction")
            res.out[sl, h] = out
            if want_traj:
                for t in range(T):
                    res.traj[(bos + t, h)] = traj[t]
            rec = cache.records.setdefault((r, h), {
                "k": np.zeros((layer.window, D)), "v": np.zeros((layer.window, D)),
                "g": np.zeros((layer.window, D)), "beta": np.zeros(layer.window),
                "delta": np.zeros((layer.window, D))})
            rec["k"][:T] = step.k[sl, h]
            rec["g"][:T] = step.g_raw[sl, h]
            if delta is not None:      # correction records: k, g_raw and the delta
                rec["delta"][:T] = delta
            else:
                rec["v"][:T] = step.v[sl, h]
                rec["beta"][:T] = step.beta_raw[sl, h]
        return b

    for item in _map_rows(run, list(rows), threads):
        if isinstance(item, RowIssue):
            res.issues.append(item)
        elif item is not None:
            res.rows_run.append(item)
    return res


def commit_len(num_accepted: int, T: int, Q: int) -> int:
    """``_prepare_commit_plan_kernel``: accepted count clamped to [0, T] and
    to the record window Q."""
    return min(max(int(num_accepted), 0), T, Q)


def commit(layer: Layer, cache: Cache, step: Step, num_accepted, *,
           deferred: bool = False, eager=None, rows=None, heads=None,
           threads: int = 1) -> list:
    """Commit after sampling (recoverssm.py commit context; context.py
    deferred commit).  Returns the list of invalid rows."""
    B = len(step.state_indices)
    H = layer.num_heads
    rows = range(B) if rows is None else rows
    heads = range(H) if heads is None else heads

    def run(b):
        T = _row_len(step.cu_seqlens, b)
        slot = int(step.state_indices[b])
        r = _record_slot(step.record_rows, b)
        bad = _row_checks(layer, cache, T, slot, r)
        if bad:
            # a deferred commit rewrites the pending count of every row whose
            # record slot is usable, a skipped row's to 0: its records now
            # hold this step's tokens, not the ones the old count replays
            if deferred and bad != "record" and r >= 0:
                cache.pending[r] = 0
            return RowIssue(b, bad)
        n = commit_len(num_accepted[b], T, layer.window)
        valid = slot > 0 and n > 0 and r >= 0
        if deferred:
            now = bool(eager[b]) if eager is not None else False
            if r >= 0:
                cache.pending[r] = n if (valid and not now) else 0
            if not now:
                return None
        if not valid:
            return None
        for h in heads:
            cache.set_state(slot, h, _replay_records(layer, cache, slot, h, r, n))
        return None

    return [x for x in _map_rows(run, list(rows), threads) if x is not None]


def flush(layer: Layer, cache: Cache, step: Step, *, rows=None, heads=None,
          threads: int = 1) -> list:
    """``KDADeferredCommitContext.flush``: fold each row's pending replay into
    its checkpoint in place; pending is left for the next commit to rewrite."""
    B = len(step.state_indices)
    H = layer.num_heads
    rows = range(B) if rows is None else rows
    heads = range(H) if heads is None else heads

    def run(b):
        slot = int(step.state_indices[b])
        r = _record_slot(step.record_rows, b)
        bad = _row_checks(layer, cache, 0, slot, r)
        if bad:
            return RowIssue(b, bad)
        if slot <= 0 or r < 0:
            return None
        p = int(cache.pending[r])
        if p < 0 or p > layer.window:
            return RowIssue(b, "pending")
        if p == 0:
            return None
        for h in heads:
            cache.set_state(slot, h, _replay_records(layer, cache, slot, h, r, p))
        return None

    return [x for x in _map_rows(run, list(rows), threads) if x is not None]


def conv_history(width: int, window: int) -> int:
    """Columns of conv history a row keeps: the conv state is
    ``history + Q - 1`` wide (the commit context derives the history length
    as the width minus the window plus one)."""
    return int(width) - int(window) + 1


def conv_compact(conv, cu_seqlens, state_indices, num_accepted, window: int):
    """Conv-state compaction of a commit (``_compact_conv_state_kernel``,
    non-align mode: the final state is the source state).

    ``conv`` is the logical conv-state pool ``[slots, conv_dim, width]`` (any
    dtype: the values are moved, not computed).  For every row b with
    T = cu_seqlens[b+1] - cu_seqlens[b], slot s = state_indices[b] and
    n = min(max(num_accepted[b], 0), T, Q): if s > 0 and n > 0, the columns
    [n - 1, n - 1 + history) of every channel of slot s are copied to columns
    [0, history), reading all of them before writing any (the kernel loads
    the whole block, then stores it).  Other rows and the columns from
    ``history`` on are left alone.  Rows with T outside [0, Q] or s beyond
    the pool are invalid: skipped and reported.

    Returns (new pool, list of RowIssue)."""
    out = np.array(conv, copy=True)
    S, _, width = out.shape
    hist = conv_history(width, window)
    if hist < 1:
        raise ValueError("conv state narrower than its window")
    issues = []
    for b in range(len(state_indices)):
        T = _row_len(cu_seqlens, b)
        slot = int(state_indices[b])
        if T < 0 or T > window:
            issues.append(RowIssue(b, "length"))
            continue
        if slot >= S:
            issues.append(RowIssue(b, "slot"))
            continue
        n = commit_len(num_accepted[b], T, window)
        if slot <= 0 or n <= 0:
            continue
        src = np.array(out[slot, :, n - 1:n - 1 + hist], copy=True)
        out[slot, :, 0:hist] = src
    return out, issues


# ---------------------------------------------------------------------------
# Align mode (paged mamba blocks)
# ---------------------------------------------------------------------------

@dataclass
class AlignPlan:
    n: int                   # commit count
    final: int               # block slot of the state after token n - 1
    boundary: int            # block slot of the state at the crossed boundary, or 0
    boundary_len: int        # tokens up to that boundary (0 when none)


def align_plan(n: int, num_computed: int, block_row, block_size: int):
    """``_prepare_commit_plan_kernel``, align branch, for a row whose commit
    count is n > 0: token t of the step sits at position num_computed + t.
    The final state belongs to the block of the last committed token,
    column (num_computed + n - 1) // block_size (the table's last column if
    it runs past the table).  The first block boundary after num_computed
    (the next multiple of block_size above it) is crossed when the step
    reaches it; the state after those boundary_len tokens belongs to the
    block that ends there.  Returns None when that block lies past the
    table."""
    width = len(block_row)
    final_col = min(max(num_computed + n - 1, 0) // block_size, width - 1)
    next_boundary = (num_computed // block_size + 1) * block_size
    boundary, boundary_len = 0, next_boundary - num_computed
    if num_computed + n >= next_boundary:
        col = next_boundary // block_size - 1
        if col >= width:
            return None
        boundary = int(block_row[col])
    return AlignPlan(n, int(block_row[final_col]), boundary, boundary_len)


def _align_row(layer, cache_slots, T, slot, num_accepted, num_computed, block_row, block_size):
    """Plan of one row, or (None, reason) / (None, None) when it commits nothing."""
    n = commit_len(num_accepted, T, layer.window)
    if slot <= 0 or n <= 0:
        return None, None
    if int(num_computed) < 0:
        return None, "block"
    plan = align_plan(n, int(num_computed), block_row, block_size)
    if plan is None:
        return None, "block"
    if plan.final >= cache_slots or plan.boundary >= cache_slots:
        return None, "slot"
    if plan.final <= 0:
        return None, None
    return plan, None


def commit_align(layer: Layer, cache: Cache, step: Step, num_accepted, block_table,
                 num_computed, block_size: int, *, request_indices=None, deferred: bool = False,
                 eager=None, rows=None, heads=None, threads: int = 1) -> list:
    """Align-mode commit (recoverssm.py commit context with a block table;
    ``_replay_indices_kernel``): each valid row replays its first n records
    from the checkpoint of ``state_indices[b]`` and writes the state after
    token n - 1 to its final block and, if the boundary comes before the last
    token (boundary_len < n), the state after boundary_len tokens to the
    boundary block.  The source slot itself is not written unless it is one
    of those blocks.  ``num_accepted``, ``num_computed`` and the block-table
    rows are indexed by request (``request_indices[b]``, or b).

    ``deferred`` (the Kimi-K3 context page's commit with a block table and
    pending / eager): a valid row whose final block is its own state slot
    and that owes no boundary block only records n as the pending replay of
    its record slot; the next verify's fold, which stores to the row's slot,
    then leaves the state after n tokens in that final block.  Every other
    valid row (an ``eager`` row, a row whose accepted tokens end in another
    block, or one that crosses a boundary before its last token) is
    committed now, and its pending count, like that of every row that
    commits nothing, is set to 0.  Returns the list of invalid rows."""
    B = len(step.state_indices)
    H = layer.num_heads
    rows = range(B) if rows is None else rows
    heads = range(H) if heads is None else heads

    def clear(r):
        if deferred and r >= 0:
            cache.pending[r] = 0

    def run(b):
        T = _row_len(step.cu_seqlens, b)
        slot = int(step.state_indices[b])
        r = _record_slot(step.record_rows, b)
        bad = _row_checks(layer, cache, T, slot, r)
        if bad:
            if bad != "record":
                clear(r)
            return RowIssue(b, bad)
        req = b if request_indices is None else int(request_indices[b])
        if req < 0 or req >= len(block_table):
            clear(r)
            return RowIssue(b, "block")
        if r < 0:  # no records: nothing to replay
            return None
        plan, bad = _align_row(layer, cache.num_slots, T, slot, num_accepted[req],
                               num_computed[req], block_table[req], block_size)
        if bad:
            clear(r)
            return RowIssue(b, bad)
        if plan is None:
            clear(r)
            return None
        mid_due = plan.boundary > 0 and plan.boundary_len < plan.n
        if deferred:
            now = (eager is not None and bool(eager[b])) or plan.final != slot or mid_due
            cache.pending[r] = 0 if now else plan.n
            if not now:
                return None
        for h in heads:
            # both replays start from the checkpoint as it was before the commit
            mid = None
            if mid_due:
                mid = _replay_records(layer, cache, slot, h, r, plan.boundary_len)
            end = _replay_records(layer, cache, slot, h, r, plan.n)
            if mid is not None:
                cache.set_state(plan.boundary, h, mid)
            cache.set_state(plan.final, h, end)
        return None

    return [x for x in _map_rows(run, list(rows), threads) if x is not None]


def conv_compact_align(conv, cu_seqlens, state_indices, num_accepted, window: int,
                       block_table, num_computed, block_size: int, *, request_indices=None):
    """Align-mode conv compaction (``_compact_conv_state_kernel`` with
    ALIGN_MODE): the window at column n - 1 of the source slot goes to
    columns [0, history) of the final block, and the window at column
    boundary_len - 1 to the boundary block when there is one; both are read
    before either is written.  Returns (new pool, list of RowIssue)."""
    out = np.array(conv, copy=True)
    S, _, width = out.shape
    hist = conv_history(width, window)
    if hist < 1:
        raise ValueError("conv state narrower than its window")
    layer = Layer(0, 0, window, None, None, False, 0.0, 1.0)
    issues = []
    for b in range(len(state_indices)):
        T = _row_len(cu_seqlens, b)
        slot = int(state_indices[b])
        if T < 0 or T > window:
            issues.append(RowIssue(b, "length"))
            continue
        if slot >= S:
            issues.append(RowIssue(b, "slot"))
            continue
        req = b if request_indices is None else int(request_indices[b])
        if req < 0 or req >= len(block_table):
            issues.append(RowIssue(b, "block"))
            continue
        plan, bad = _align_row(layer, S, T, slot, num_accepted[req], num_computed[req],
                               block_table[req], block_size)
        if bad:
            issues.append(RowIssue(b, bad))
            continue
        if plan is None:
            continue
        fin = np.array(out[slot, :, plan.n - 1:plan.n - 1 + hist], copy=True)
        bnd = None
        if plan.boundary > 0:
            bnd = np.array(out[slot, :, plan.boundary_len - 1:plan.boundary_len - 1 + hist],
                           copy=True)
        if bnd is not None:
            out[plan.boundary, :, 0:hist] = bnd
        out[plan.final, :, 0:hist] = fin
    return out, issues


def record_state_blocks(idx_mapping, num_sampled, num_computed, state_column, num_accepted,
                        block_size: int, block_table_width: int, *, num_rows=None,
                        request_indices=None):
    """Align-mode bookkeeping after a commit (recoverssm.py,
    ``_record_state_block_kernel`` and ``record_state_blocks``): each spec
    row's request q (``request_indices[i]``, or i) has a slot s =
    ``idx_mapping[q]`` in the running arrays; s < 0 means nothing to record.
    Its last committed token sits at position max(num_computed[q] +
    num_sampled[q] - 1, 0); ``state_column[s]`` becomes the block-table
    column holding it (the last column when it runs past the table) and
    ``num_accepted[s]`` becomes 1.  Rows whose q lies outside the request
    arrays ("block") or whose s lies outside the running arrays ("slot")
    are skipped (this build's reading; the page checks neither).  Returns
    (state_column, num_accepted, list of RowIssue) as new arrays."""
    col = np.array(state_column, dtype=np.int64, copy=True)
    acc = np.array(num_accepted, dtype=np.int64, copy=True)
    if num_rows is not None:
        n_rows = num_rows
    else:
        n_rows = len(idx_mapping) if request_indices is None else len(request_indices)
    issues = []
    for i in range(n_rows):
        q = i if request_indices is None else int(request_indices[i])
        if q < 0 or q >= len(idx_mapping):
            issues.append(RowIssue(i, "block"))
            continue
        s = int(idx_mapping[q])
        if s < 0:
            continue
        if s >= len(col):
            issues.append(RowIssue(i, "slot"))
            continue
        last = max(int(num_computed[q]) + int(num_sampled[q]) - 1, 0)
        col[s] = min(last // block_size, block_table_width - 1)
        acc[s] = 1
    return col, acc, issues


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)
