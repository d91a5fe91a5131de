"""GPU check of the benchmark's end-to-end pipeline (bench.HostIO).

The end-to-end figure counts only if its steps do the work: every step's
inputs reach the device from pinned host memory, and its outputs come back
after the step computed them, before a later step overwrites them.  Issued
call by call from the host, and replayed from the captured CUDA graph, the
outputs copied back must equal, bit for bit, those of the same steps run on
the device alone.  The state pools rotate, so consecutive steps differ and a
copy taken at the wrong time would show.
"""

import pytest
import torch

import bench
from linear_attention_speculative_kda_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture
def two_pools(monkeypatch):
    wl = W.generate("tiny")
    # two pool copies: consecutive steps read different checkpoints, and the
    # captured graph holds 8 steps
    monkeypatch.setattr(bench, "POOL_ROTATION_BYTES", 2 * wl.pool.numel() * 4)
    return wl


def _reference(wl, k_steps):
    eng = bench.Engine(wl, torch.device("cuda", 0))
    outs = []
    for _ in range(k_steps):
        eng.run_step(steps=eng.steps)
        torch.cuda.synchronize()
        outs.append([st["out"].cpu().clone() for st in eng.steps])
    assert int(eng.err.item()) == 0
    return outs


def _check(hio, ref, last_step):
    # the last step on each input set: last_step (its parity) and last_step - 1
    for j in (last_step - 1, last_step):
        for got, want in zip(hio.h_out[j & 1], ref[j]):
            assert torch.equal(got, want), j
    for dev_set in hio.sets:
        for st, ins in zip(dev_set, hio.h_in):
            for key, host in ins.items():
                assert torch.equal(st[key].cpu(), host), key


def test_host_issued_steps_copy_the_right_outputs(two_pools):
    wl = two_pools
    ref = _reference(wl, 6)
    eng = bench.Engine(wl, torch.device("cuda", 0))
    assert len(eng.pools) == 2
    hio = bench.HostIO(eng)
    hio.run(6)
    torch.cuda.synchronize()
    assert int(eng.err.item()) == 0
    _check(hio, ref, 5)


def test_graph_replayed_steps_copy_the_right_outputs(two_pools):
    wl = two_pools
    eng = bench.Engine(wl, torch.device("cuda", 0))
    hio = bench.HostIO(eng)
    n = hio.graph_steps()
    assert n == 8
    ref = _reference(wl, 2 * n)
    graph = hio.capture()
    hio.fill_first()
    graph.replay()
    torch.cuda.synchronize()
    assert int(eng.err.item()) == 0
    _check(hio, ref, n - 1)
    graph.replay()  # the next 8 steps: the pools keep rotating
    torch.cuda.synchronize()
    _check(hio, ref, 2 * n - 1)
    del graph
