"""GPU parity at the largest head count the library supports (32767).

A work item carries its head in the top half of a 32-bit word, and the grid
covers B * H tiles, so the last heads of a 32767-head layer are the edge of
both.  The buffers are generated on the device (a 4.3 GB state pool); the
oracle checks a sample of heads, as a sub-problem of those heads alone
(heads are independent): the first, a middle one and the last two.
"""

import numpy as np
import pytest
import torch

from linear_attention_speculative_kda_gb300 import api
from oracle import kda_oracle as O
from tests.helpers import assert_out_close, assert_state_close

pytestmark = pytest.mark.gpu

H = 32767
D = 128


def _f64(t):
    return t.detach().float().cpu().double().numpy()


@pytest.mark.parametrize("Q,T,bounded", [(2, 2, False), (8, 6, True)])
def test_max_heads_verify_and_commit(Q, T, bounded):
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev)
    gen.manual_seed(1000 + Q)
    S = 2  # slot 0 is the null slot
    pool = torch.randn((S, H, D, D), generator=gen, device=dev) * 0.1
    heads = [0, 12345, H - 2, H - 1]
    hs = torch.tensor(heads, device=dev)
    sub_pool = np.zeros((S, len(heads), D, D), np.float32)
    sub_pool[1] = pool[1][hs].cpu().numpy()  # the sampled checkpoints, before the launches
    A_log = torch.rand((H,), generator=gen, device=dev) * 2.0 - 1.0
    g_bias = torch.randn((H * D,), generator=gen, device=dev) * 0.1
    qkv = torch.randn((T, 3, H, D), generator=gen, device=dev).to(torch.bfloat16)
    g_raw = torch.randn((T, H, D), generator=gen, device=dev).to(torch.bfloat16)
    beta_raw = torch.randn((T, H), generator=gen, device=dev).to(torch.bfloat16)
    cu = torch.tensor([0, T], dtype=torch.int32, device=dev)
    slots = torch.tensor([1], dtype=torch.int32, device=dev)
    acc = torch.tensor([T - 1], dtype=torch.int32, device=dev)
    records = api.allocate_records(H, Q, 1, dev)
    out = torch.empty((T, H, D), dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lb = -5.0 if bounded else None
    api.kda_verify(qkv[:, 0], qkv[:, 1], qkv[:, 2], g_raw, beta_raw, A_log, g_bias, pool, cu,
                   slots, records, out, window=Q, record_slots=1, lower_bound=lb,
                   error_word=err)
    api.kda_commit(A_log, g_bias, pool, cu, slots, acc, records, window=Q, record_slots=1,
                   lower_bound=lb, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    layer = O.Layer(len(heads), D, Q, _f64(A_log[hs]), _f64(g_bias.view(H, D)[hs]), bounded,
                    lb if bounded else 0.0, D ** -0.5)
    step = O.Step(_f64(qkv[:, 0][:, hs]), _f64(qkv[:, 1][:, hs]), _f64(qkv[:, 2][:, hs]),
                  _f64(g_raw[:, hs]), _f64(beta_raw[:, hs]), np.array([0, T], np.int32),
                  np.array([1], np.int32))
    cache = O.Cache(sub_pool, 1)
    res = O.verify(layer, cache, step)
    assert O.commit(layer, cache, step, np.array([T - 1])) == []
    assert_out_close(out[:, hs], res.out)
    for i in range(len(heads)):
        assert_state_close(pool[1, heads[i]].double().cpu().numpy(), cache.written[(1, i)])


def test_deferred_chain_beyond_the_balanced_plan_rows():
    """4500 rows, more than the 4096 the commits' balanced plan takes: the
    deferred commits fall back to the strided plan, where each row's pending
    count is written by the CTA that plans the row's head 0.  Two deferred
    steps (a fold in the second verify), checked on sampled rows, the last
    ones among them, against the oracle: outputs, stored states and pending
    counts."""
    from linear_attention_speculative_kda_gb300 import workloads as W
    from tests.helpers import DeviceRun, oracle_cache, oracle_layer, oracle_step

    B = 4500
    lens = np.random.default_rng(5).integers(0, 3, size=B).tolist()
    wl = W.custom(B=B, H=2, Q=2, lens=lens, S=B + 2, R=B + 4, deferred=True, steps=2,
                  seed=77, eager_prob=0.3)
    g = DeviceRun(wl, sentinel=False)
    g.verify(0, pending=True)
    g.commit(0, deferred=True)
    g.verify(1, pending=True)
    g.commit(1, deferred=True)
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    rng = np.random.default_rng(9)
    rows = sorted(set(rng.choice(B, size=20, replace=False).tolist()) | {4095, 4096, 4097, B - 1})
    layer, cache = oracle_layer(wl), oracle_cache(wl)
    s1, s2 = oracle_step(wl, 0), oracle_step(wl, 1)
    O.verify(layer, cache, s1, pending=True, rows=rows)
    O.commit(layer, cache, s1, wl.steps[0].num_accepted.numpy(), deferred=True,
             eager=wl.steps[0].eager.numpy(), rows=rows)
    r2 = O.verify(layer, cache, s2, pending=True, rows=rows)
    O.commit(layer, cache, s2, wl.steps[1].num_accepted.numpy(), deferred=True,
             eager=wl.steps[1].eager.numpy(), rows=rows)
    assert_out_close(g.out, r2.out)
    pool = g.pool.cpu()
    for (slot, h), ref in cache.written.items():
        assert_state_close(pool[slot, h].double().numpy(), ref)
    pending = g.pending.cpu().numpy()
    rr = wl.record_rows.numpy()
    for b in rows:
        assert pending[rr[b]] == cache.pending[rr[b]], b
