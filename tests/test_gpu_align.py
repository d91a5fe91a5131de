"""GPU parity of the align-mode commit and conv compaction (paged blocks)
against the oracle, and bit-exactness of the stored blocks against the GPU
verify trajectory.  Tolerances as in test_gpu_parity: fp32 states normwise
1e-5 per tile against the oracle; the stored states bit-identical to the
trajectory the verify computed; conv windows bit-identical."""

import numpy as np
import pytest
import torch

from linear_attention_speculative_kda_gb300 import api
from linear_attention_speculative_kda_gb300 import workloads as W
from oracle import kda_oracle as O
from tests.helpers import DeviceRun, assert_state_close, oracle_cache, oracle_layer, oracle_step

pytestmark = pytest.mark.gpu

WIDTH = 6


def _case(Q, bounded=False, seed=40, B=8):
    lens = [Q, Q, max(1, Q - 1), Q, 2 if Q >= 2 else 1, Q, Q, 1][:B]
    sources = list(range(1, B + 1))
    sources[3] = 0                                     # a null row
    S = 1 + B + B * WIDTH
    kw = dict(bounded=True, lower_bound=-5.0) if bounded else {}
    wl = W.custom(B=B, H=2, Q=Q, lens=lens, S=S, seed=seed, slots=sources, **kw)
    rng = np.random.default_rng(seed)
    # request b owns blocks 1 + B + b*WIDTH .. ; a permuted request order
    table = (1 + B + np.arange(B * WIDTH)).reshape(B, WIDTH).astype(np.int32)
    bs = max(Q, 4)
    num_computed = rng.integers(0, bs * (WIDTH - 1), size=B).astype(np.int32)
    return wl, table, num_computed, bs


def _run_align(g, wl, table, nc, bs, request_indices=None, acc=None):
    d = g.dev
    i32 = dict(dtype=torch.int32, device=d)
    acc = g.steps[0]["num_accepted"] if acc is None else torch.tensor(acc, **i32)
    api.kda_commit_align(g.A_log, g.g_bias, g.pool, g.cu, g.slots, acc, g.records,
                         torch.tensor(table, **i32), torch.tensor(nc, **i32), block_size=bs,
                         request_indices=None if request_indices is None
                         else torch.tensor(request_indices, **i32),
                         record_rows=g.record_rows, error_word=g.err, **g.kw())
    torch.cuda.synchronize()


@pytest.mark.parametrize("Q,bounded", [(4, False), (8, False), (8, True), (1, False)])
def test_commit_align_against_oracle_and_trajectory(Q, bounded):
    wl, table, nc, bs = _case(Q, bounded, seed=40 + Q)
    g = DeviceRun(wl, with_traj=True)
    g.verify()
    torch.cuda.synchronize()
    traj = g.traj.clone()
    _run_align(g, wl, table, nc, bs)
    assert int(g.err.item()) == 0
    layer, step = oracle_layer(wl), oracle_step(wl)
    cache = oracle_cache(wl)
    O.verify(layer, cache, step)
    acc = wl.steps[0].num_accepted.numpy()
    assert O.commit_align(layer, cache, step, acc, table, nc, bs) == []
    pool = g.pool.cpu().numpy()
    cu = wl.cu_seqlens.numpy()
    written = set(cache.written)
    for (slot, h), ref in cache.written.items():
        assert_state_close(pool[slot, h].astype(np.float64), ref)
    # bit-exact against the trajectory at the final and boundary tokens
    tr = traj.cpu()
    for b in range(wl.spec.B):
        slot = int(wl.state_indices[b])
        n = O.commit_len(acc[b], cu[b + 1] - cu[b], Q)
        if slot <= 0 or n <= 0:
            continue
        plan = O.align_plan(n, int(nc[b]), table[b], bs)
        for h in range(wl.spec.H):
            assert torch.equal(g.pool[plan.final, h].cpu(), tr[cu[b] + n - 1, h])
            if plan.boundary > 0 and plan.boundary_len < n:
                assert torch.equal(g.pool[plan.boundary, h].cpu(),
                                   tr[cu[b] + plan.boundary_len - 1, h])
    # everything else, the sources included, is untouched
    pool0 = g.pool0.cpu().numpy()
    for slot in range(pool.shape[0]):
        for h in range(wl.spec.H):
            if (slot, h) not in written:
                assert np.array_equal(pool[slot, h], pool0[slot, h])


def test_blocks_at_source_equal_the_plain_commit():
    wl, _, nc, bs = _case(4, seed=50)
    table = np.repeat(wl.state_indices.numpy()[:, None], WIDTH, axis=1).astype(np.int32)
    a, p = DeviceRun(wl), DeviceRun(wl)
    a.verify()
    p.verify()
    _run_align(a, wl, table, nc, bs)
    p.commit()
    torch.cuda.synchronize()
    assert int(a.err.item()) == 0 and int(p.err.item()) == 0
    assert torch.equal(a.pool, p.pool)


def test_request_indices_permute_the_tables():
    wl, table, nc, bs = _case(4, seed=51)
    B = wl.spec.B
    perm = np.random.default_rng(1).permutation(B).astype(np.int32)
    # request perm[b] holds row b's table, count and accepted tokens
    table_p = np.zeros_like(table)
    nc_p = np.zeros_like(nc)
    acc = wl.steps[0].num_accepted.numpy()
    acc_p = np.zeros_like(acc)
    table_p[perm] = table
    nc_p[perm] = nc
    acc_p[perm] = acc
    a, p = DeviceRun(wl), DeviceRun(wl)
    a.verify()
    p.verify()
    _run_align(a, wl, table, nc, bs)
    _run_align(p, wl, table_p, nc_p, bs, request_indices=perm, acc=acc_p.tolist())
    assert int(a.err.item()) == 0 and int(p.err.item()) == 0
    assert torch.equal(a.pool, p.pool)


def test_bad_blocks_are_flagged_and_skipped():
    wl, table, nc, bs = _case(4, seed=52)
    table = table.copy()
    nc = nc.copy()
    S = wl.spec.S
    table[0, :] = S + 5                      # final block past the pool
    nc[1] = bs * WIDTH + bs - 1              # boundary block past the table
    g = DeviceRun(wl)
    g.verify()
    acc = np.full(wl.spec.B, 2, dtype=np.int32)
    _run_align(g, wl, table, nc, bs, acc=acc.tolist())
    assert int(g.err.item()) == (api.ROW_BAD_SLOT | api.ROW_BAD_BLOCK)
    layer, step = oracle_layer(wl), oracle_step(wl)
    cache = oracle_cache(wl)
    O.verify(layer, cache, step)
    issues = O.commit_align(layer, cache, step, acc, table, nc, bs)
    assert {(i.row, i.reason) for i in issues} == {(0, "slot"), (1, "block")}
    pool = g.pool.cpu().numpy()
    for (slot, h), ref in cache.written.items():
        assert_state_close(pool[slot, h].astype(np.float64), ref)


@pytest.mark.parametrize("layout", ["dim_first", "col_first"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_conv_compact_align_bit_exact(layout, dtype):
    rng = np.random.default_rng(60)
    Q, B, C, bs = 4, 9, 200, 4
    width_bt = 5
    S = 1 + B + B * width_bt
    conv_w = 3 + Q - 1
    conv = W.conv_state(S, C, conv_w, dtype=dtype, seed=61, layout=layout)
    lens = rng.integers(0, Q + 1, size=B)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    slots = np.arange(1, B + 1, dtype=np.int32)
    slots[2] = 0
    table = (1 + B + np.arange(B * width_bt)).reshape(B, width_bt).astype(np.int32)
    nc = rng.integers(0, bs * (width_bt - 1), size=B).astype(np.int32)
    acc = rng.integers(-1, Q + 2, size=B).astype(np.int32)
    dev = torch.device("cuda:0")
    if layout == "dim_first":
        dconv = conv.to(dev)
    else:
        dconv = conv.transpose(1, 2).contiguous().to(dev).transpose(1, 2)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    t = lambda a: torch.tensor(a, dtype=torch.int32, device=dev)  # noqa: E731
    api.kda_conv_compact_align(dconv, t(cu), t(slots), t(acc), t(table), t(nc), block_size=bs,
                               window=Q, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    bits = {torch.bfloat16: torch.int16, torch.float32: torch.int32}[dtype]
    raw = conv.contiguous().view(bits).numpy()
    want, issues = O.conv_compact_align(raw, cu, slots, acc, Q, table, nc, bs)
    assert issues == []
    got = dconv.cpu().contiguous().view(bits).numpy()
    assert np.array_equal(got, want)


def test_full_size_align_commit():
    """deferred2's rows at full size (1024 requests x 16 heads) with two
    blocks per request, as the benchmark runs the align commit: every stored
    block equals the verify trajectory bit for bit, and a sample of tiles is
    checked against the oracle."""
    wl = W.generate("deferred2", pool=False)
    sp = wl.spec
    B, H, D, width, bs = sp.B, sp.H, sp.D, 2, 16
    S = 1 + B + B * width
    gen = torch.Generator().manual_seed(3)
    pool_cpu = torch.randn((S, H, D, D), generator=gen) * 0.05
    sources = torch.where(wl.state_indices > 0, torch.arange(1, B + 1, dtype=torch.int32),
                          torch.zeros(B, dtype=torch.int32))
    wl.pool = pool_cpu
    wl.state_indices = sources
    wl.spec = W.Spec(**{**sp.__dict__, "S": S})
    table = (1 + B + np.arange(B * width)).reshape(B, width).astype(np.int32)
    nc = torch.randint(0, bs, (B,), generator=gen, dtype=torch.int32).numpy()
    g = DeviceRun(wl, with_traj=True, sentinel=False)
    g.verify()
    torch.cuda.synchronize()
    _run_align(g, wl, table, nc, bs)
    assert int(g.err.item()) == 0
    acc = wl.steps[0].num_accepted.numpy()
    cu = wl.cu_seqlens.numpy()
    fin_s, fin_t, mid_s, mid_t = [], [], [], []
    for b in range(B):
        n = O.commit_len(int(acc[b]), cu[b + 1] - cu[b], sp.Q)
        if int(sources[b]) <= 0 or n <= 0:
            continue
        plan = O.align_plan(n, int(nc[b]), table[b], bs)
        fin_s.append(plan.final)
        fin_t.append(int(cu[b]) + n - 1)
        if plan.boundary > 0 and plan.boundary_len < n:
            mid_s.append(plan.boundary)
            mid_t.append(int(cu[b]) + plan.boundary_len - 1)
    assert fin_s and mid_s
    dev = g.pool.device
    assert torch.equal(g.pool[torch.tensor(fin_s, device=dev)], g.traj[torch.tensor(fin_t, device=dev)])
    assert torch.equal(g.pool[torch.tensor(mid_s, device=dev)], g.traj[torch.tensor(mid_t, device=dev)])
    # a sample against the oracle
    rng = np.random.default_rng(0)
    rows = sorted(rng.choice(B, size=16, replace=False).tolist())
    heads = sorted(rng.choice(H, size=2, replace=False).tolist())
    layer, step = oracle_layer(wl), oracle_step(wl)
    cache = oracle_cache(wl)
    O.verify(layer, cache, step, rows=rows, heads=heads)
    assert O.commit_align(layer, cache, step, acc, table, nc, bs, rows=rows, heads=heads) == []
    assert cache.written
    for (slot, h), ref in cache.written.items():
        assert_state_close(g.pool[slot, h].double().cpu().numpy(), ref)


def _deferred_align_case(Q, bounded, seed):
    """Rows whose state slot is the block of their last computed token (the
    table column (c - 1) // bs, as a runner keeps it), so that the deferred
    form defers the rows that stay in their block."""
    B = 12
    lens = [Q, Q, max(1, Q - 1), Q, min(2, Q), Q, Q, 1, Q, Q, max(1, Q - 2), Q]
    kw = dict(bounded=True, lower_bound=-5.0) if bounded else {}
    wl = W.custom(B=B, H=2, Q=Q, lens=lens, S=1 + B + B * WIDTH, seed=seed,
                  slots=list(range(1, B + 1)), **kw)
    rng = np.random.default_rng(seed)
    bs = max(Q, 4) * 2
    nc = rng.integers(1, bs * (WIDTH - 1), size=B).astype(np.int32)
    table = (1 + B + np.arange(B * WIDTH)).reshape(B, WIDTH).astype(np.int32)
    for b in range(B):
        table[b, (nc[b] - 1) // bs] = int(wl.state_indices[b])
    eager = (rng.random(B) < 0.25).astype(np.uint8)
    return wl, table, nc, bs, eager


@pytest.mark.parametrize("Q,bounded", [(4, False), (8, True)])
def test_deferred_align_commit_against_oracle_and_eager(Q, bounded):
    """The deferred align commit: pending counts equal the oracle's, the rows
    committed now match the oracle and the eager align commit bit for bit, and
    after a flush the whole pool equals the eager align commit's."""
    wl, table, nc, bs, eager = _deferred_align_case(Q, bounded, seed=60 + Q)
    d = torch.device("cuda")
    i32 = dict(dtype=torch.int32, device=d)
    acc = wl.steps[0].num_accepted.numpy()
    e, g = DeviceRun(wl), DeviceRun(wl)
    for run in (e, g):
        run.verify()
    _run_align(e, wl, table, nc, bs)
    g.pending.fill_(7)
    api.kda_commit_align(g.A_log, g.g_bias, g.pool, g.cu, g.slots, g.steps[0]["num_accepted"],
                         g.records, torch.tensor(table, **i32), torch.tensor(nc, **i32),
                         block_size=bs, record_rows=g.record_rows, pending=g.pending,
                         eager=torch.tensor(eager, dtype=torch.uint8, device=d),
                         error_word=g.err, **g.kw())
    torch.cuda.synchronize()
    assert int(e.err.item()) == 0 and int(g.err.item()) == 0
    layer, step = oracle_layer(wl), oracle_step(wl)
    cache = oracle_cache(wl)
    O.verify(layer, cache, step)
    cache.pending[:] = 7
    cache.written.clear()
    assert O.commit_align(layer, cache, step, acc, table, nc, bs, deferred=True,
                          eager=eager) == []
    assert g.pending.cpu().tolist() == cache.pending.tolist()
    deferred = [b for b in range(wl.spec.B) if cache.pending[b] > 0]
    assert deferred and len(deferred) < wl.spec.B     # both kinds occur
    pool = g.pool.cpu()
    for (slot, h), ref in cache.written.items():
        assert_state_close(pool[slot, h].double().numpy(), ref)
        assert torch.equal(pool[slot, h], e.pool[slot, h].cpu())
    # the deferred rows' slots still hold the checkpoint until the fold
    for b in deferred:
        s = int(wl.state_indices[b])
        assert torch.equal(g.pool[s], g.pool0[s])
    g.flush()
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    assert torch.equal(g.pool, e.pool)


@pytest.mark.parametrize("with_indices", [False, True], ids=["rows_are_requests", "request_indices"])
def test_record_state_blocks_bit_exact(with_indices):
    """kda_record_state_blocks against the oracle, bit for bit: 700 requests
    (three CTAs and a ragged tail), a third of them without a running slot,
    columns past the table clamped; through request_indices, a permuted
    subset of the requests, plus one request index and one slot out of range
    (flagged, skipped)."""
    rng = np.random.default_rng(21 if with_indices else 20)
    dev = torch.device("cuda", 0)
    R, S, bs, width = 700, 900, 16, 8
    idx = rng.permutation(S)[:R].astype(np.int32)
    idx[rng.random(R) < 0.33] = -1
    nc = rng.integers(0, 150, size=R).astype(np.int32)
    ns = rng.integers(0, 9, size=R).astype(np.int32)
    req = None
    if with_indices:
        req = rng.permutation(R)[:500].astype(np.int32)
        req[7] = R + 3                      # past the requests: KDA_ROW_BAD_BLOCK
        idx[req[11]] = S + 5                # past the running slots: KDA_ROW_BAD_SLOT
    col0 = rng.integers(0, 99, size=S).astype(np.int32)
    acc0 = rng.integers(2, 9, size=S).astype(np.int32)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    col, acc, err = t(col0), t(acc0), torch.zeros(1, dtype=torch.int32, device=dev)
    api.kda_record_state_blocks(t(idx), t(ns), t(nc), col, acc, block_size=bs,
                                block_table_width=width,
                                request_indices=None if req is None else t(req), error_word=err)
    torch.cuda.synchronize()
    want_col, want_acc, issues = O.record_state_blocks(idx, ns, nc, col0, acc0, bs, width,
                                                       request_indices=req)
    assert col.cpu().numpy().tolist() == want_col.tolist()
    assert acc.cpu().numpy().tolist() == want_acc.tolist()
    want_err = 0
    for i in issues:
        want_err |= api.ROW_BAD_BLOCK if i.reason == "block" else api.ROW_BAD_SLOT
    assert int(err.item()) == want_err
    assert want_err == ((api.ROW_BAD_BLOCK | api.ROW_BAD_SLOT) if with_indices else 0)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_conv_compact_align_blocks_at_the_source(dtype):
    """Channel-major pools (the 16-byte unit form of the kernel) whose block
    tables name the row's own source slot for some columns: the final block,
    the boundary block or both can be the source, and every window must still
    come from the source as it was before the call."""
    rng = np.random.default_rng(70)
    Q, B, C, bs = 4, 12, 256, 4
    width_bt = 4
    S = 1 + B + B * width_bt
    conv_w = 3 + Q - 1
    conv = W.conv_state(S, C, conv_w, dtype=dtype, seed=71)
    lens = np.full(B, Q)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    slots = np.arange(1, B + 1, dtype=np.int32)
    table = (1 + B + np.arange(B * width_bt)).reshape(B, width_bt).astype(np.int32)
    for b in range(0, B, 2):
        table[b, (b // 2) % width_bt] = slots[b]     # one column is the row's own slot
    table[1, :] = slots[1]                            # every block of row 1 is its slot
    nc = rng.integers(0, bs * (width_bt - 1), size=B).astype(np.int32)
    acc = rng.integers(1, Q + 1, size=B).astype(np.int32)
    dev = torch.device("cuda:0")
    dconv = conv.to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    t = lambda a: torch.tensor(a, dtype=torch.int32, device=dev)  # noqa: E731
    api.kda_conv_compact_align(dconv, t(cu), t(slots), t(acc), t(table), t(nc), block_size=bs,
                               window=Q, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    bits = {torch.bfloat16: torch.int16, torch.float32: torch.int32}[dtype]
    raw = conv.contiguous().view(bits).numpy()
    want, issues = O.conv_compact_align(raw, cu, slots, acc, Q, table, nc, bs)
    assert issues == []
    assert np.array_equal(dconv.cpu().contiguous().view(bits).numpy(), want)
