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
