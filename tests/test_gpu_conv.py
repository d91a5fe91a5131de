"""GPU parity of the conv-state compaction (``kda_conv_compact``) against the
oracle.  The compaction moves values, so the comparison is bit for bit, on
the raw bits of the pool, for both element sizes and both layouts."""

import numpy as np
import pytest
import torch

from linear_attention_speculative_kda_gb300 import api
from linear_attention_speculative_kda_gb300 import workloads as W
from oracle import kda_oracle as O

pytestmark = pytest.mark.gpu

BITS = {torch.bfloat16: torch.int16, torch.float32: torch.int32}


def _bits(conv: torch.Tensor) -> np.ndarray:
    """Logical [S, C, W] array of the raw element bits (exact)."""
    return conv.detach().cpu().contiguous().view(BITS[conv.dtype]).numpy()


def _run(conv_cpu, cu, slots, acc, Q):
    dev = torch.device("cuda:0")
    if conv_cpu.stride(2) == 1:
        conv = conv_cpu.to(dev)
    else:  # keep the column-major storage on the device
        conv = conv_cpu.transpose(1, 2).contiguous().to(dev).transpose(1, 2)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    i32 = dict(dtype=torch.int32, device=dev)
    api.kda_conv_compact(conv, torch.tensor(cu, **i32), torch.tensor(slots, **i32),
                         torch.tensor(acc, **i32), window=Q, error_word=err)
    torch.cuda.synchronize()
    return conv, int(err.item())


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("layout", ["dim_first", "col_first"])
@pytest.mark.parametrize("Q,kernel", [(1, 4), (4, 4), (8, 4), (3, 2), (8, 9)])
@pytest.mark.parametrize("C", [300, 512])
def test_small_ragged(dtype, layout, Q, kernel, C):
    # C = 300 leaves ragged tails and, for some widths, channels whose bytes
    # do not make 16-byte units: together the cases reach the staged, the
    # column-vector and the element-wise forms of the kernel
    rng = np.random.default_rng(Q * 10 + kernel + C)
    B, S = 11, 16
    width = kernel - 1 + Q - 1
    conv = W.conv_state(S, C, width, dtype=dtype, seed=Q + kernel, layout=layout)
    lens = rng.integers(0, Q + 1, size=B)
    lens[0] = Q
    cu = np.concatenate([[0], np.cumsum(lens)]).tolist()
    slots = rng.permutation(np.arange(1, S))[:B].tolist()
    slots[3] = 0                                   # a null row
    acc = [int(x) for x in rng.integers(-1, Q + 3, size=B)]
    got, err = _run(conv, cu, slots, acc, Q)
    assert err == 0
    want, issues = O.conv_compact(_bits(conv), cu, slots, acc, Q)
    assert issues == []
    assert np.array_equal(_bits(got), want)


def test_invalid_rows_flagged_and_skipped():
    Q, S, C, width = 4, 6, 64, 6
    conv = W.conv_state(S, C, width, seed=9)
    cu = [0, 5, 9, 13]          # row 0: T = 5 > Q
    slots = [1, 9, 2]           # row 1: slot 9 >= S
    acc = [2, 2, 3]
    got, err = _run(conv, cu, slots, acc, Q)
    assert err == (api.ROW_BAD_LENGTH | api.ROW_BAD_SLOT)
    want, issues = O.conv_compact(_bits(conv), cu, slots, acc, Q)
    assert [(i.row, i.reason) for i in issues] == [(0, "length"), (1, "slot")]
    assert np.array_equal(_bits(got), want)


def test_empty_batch():
    dev = torch.device("cuda:0")
    conv = W.conv_state(3, 8, 6).to(dev)
    before = conv.clone()
    e = torch.zeros(0, dtype=torch.int32, device=dev)
    api.kda_conv_compact(conv, torch.zeros(1, dtype=torch.int32, device=dev), e, e, window=4)
    torch.cuda.synchronize()
    assert torch.equal(conv, before)


def test_more_rows_than_one_grid_dimension():
    # 70,000 rows: the kernel strides over rows beyond the 65,535 grid limit
    Q, B, C, width = 2, 70000, 4, 4
    S = B + 1
    conv = W.conv_state(S, C, width, seed=11)
    rng = np.random.default_rng(12)
    cu = np.arange(0, 2 * B + 1, 2).tolist()
    slots = (rng.permutation(B) + 1).tolist()
    acc = rng.integers(0, 3, size=B).tolist()
    got, err = _run(conv, cu, slots, acc, Q)
    assert err == 0
    want, _ = O.conv_compact(_bits(conv), cu, slots, acc, Q)
    assert np.array_equal(_bits(got), want)


@pytest.mark.parametrize("name", ["deferred2", "mixed"])
def test_full_size_workload(name):
    wl = W.generate(name, pool=False)
    S, C, width = W.conv_shape(wl.spec)
    conv = W.conv_state(S, C, width, seed=5)
    cu = wl.cu_seqlens.tolist()
    slots = wl.state_indices.tolist()
    acc = wl.steps[0].num_accepted.tolist()
    got, err = _run(conv, cu, slots, acc, wl.spec.Q)
    assert err == 0
    want, _ = O.conv_compact(_bits(conv), cu, slots, acc, wl.spec.Q)
    assert np.array_equal(_bits(got), want)
