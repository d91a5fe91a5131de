"""Host-side logic of bench.py on CPU: the multi-rank reductions (world size 2
over gloo), the per-rank seeds of weak scaling, the algorithmic byte count,
the clock-sample summary and the profile lookup."""

import json
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from linear_attention_speculative_kda_gb300 import workloads as W  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mx = bench.max_over_ranks(10.0 + rank, world, torch.device("cpu"))
        sm = bench.sum_over_ranks(100.0 * (rank + 1), world, torch.device("cpu"))
        out.put((rank, mx, sm, bench.shard_seed(0, rank)))
    finally:
        dist.destroy_process_group()


def test_two_rank_reductions_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r[1] for r in res] == [11.0, 11.0]          # max over ranks
    assert [r[2] for r in res] == [300.0, 300.0]        # sum over ranks
    assert res[0][3] != res[1][3]                       # each rank its own batch


def test_single_rank_reductions_are_identity():
    assert bench.max_over_ranks(3.5, 1, None) == 3.5
    assert bench.sum_over_ranks(7.0, 1, None) == 7.0


def _bytes_by_loops(wl, tok=2052, rec=770):
    """Per-row loop of the algorithmic byte count: the state tile read once per
    live row, `tok` bytes per verified token (raw records: q, k, v, g_raw
    read, 2 bytes of beta, 256 of output, 770 of record written), and `rec`
    bytes per replayed record token on top of a commit's state read and
    write, counted one row at a time."""
    sp = wl.spec
    lens = (wl.cu_seqlens[1:] - wl.cu_seqlens[:-1]).tolist()
    slots = wl.state_indices.tolist()
    state = 65536

    def n_of(acc, T):
        return min(max(acc, 0), T, sp.Q)

    if not sp.deferred:
        acc = wl.steps[0].num_accepted.tolist()
        v = c = 0
        for b in range(sp.B):
            if slots[b] > 0 and lens[b] > 0:
                v += state + lens[b] * tok
            n = n_of(acc[b], lens[b])
            if slots[b] > 0 and n > 0:
                c += 2 * state + n * rec
        return [v * sp.H, c * sp.H]
    a1 = wl.steps[0].num_accepted.tolist()
    a2 = wl.steps[1].num_accepted.tolist()
    eg = wl.steps[0].eager.tolist()
    v1 = c1 = v2 = c2 = 0
    for b in range(sp.B):
        live = slots[b] > 0
        n1, n2 = n_of(a1[b], lens[b]), n_of(a2[b], lens[b])
        if live and lens[b] > 0:
            v1 += state + lens[b] * tok
        if live and n1 > 0 and eg[b]:
            c1 += 2 * state + n1 * rec
        pend = n1 if (live and n1 > 0 and not eg[b]) else 0
        if live and (lens[b] > 0 or pend > 0):
            v2 += state + lens[b] * tok + (state + pend * rec if pend else 0)
        if live and n2 > 0:
            c2 += 2 * state + n2 * rec
    return [x * sp.H for x in (v1, c1, v2, c2)]


@pytest.mark.parametrize("name", ["tiny", "dflash7"])
def test_plan_bytes_small(name):
    wl = W.generate(name)
    assert [b for _, b in bench.plan_bytes(wl)] == _bytes_by_loops(wl)


def test_plan_bytes_deferred():
    wl = W.custom(B=32, H=3, Q=4, lens=[4] * 30 + [0, 2], S=40, R=36, deferred=True, steps=2,
                  seed=5, slots=[0] * 3 + list(range(4, 33)))
    names = [n for n, _ in bench.plan_bytes(wl)]
    assert names == ["verify", "commit_deferred", "verify_fused", "commit"]
    assert [b for _, b in bench.plan_bytes(wl)] == _bytes_by_loops(wl)
    assert bench.units_per_step(wl) == 2 * 32 * 3


def test_plan_bytes_correction_records():
    # correction records: 1024 bytes per token (fp32 delta, bf16 k and g_raw)
    # written by the verify and read by a replay; a verified token then moves
    # 4 * 256 + 2 + 256 + 1024 bytes
    wl = W.custom(B=32, H=3, Q=4, lens=[4] * 30 + [0, 2], S=40, R=36, deferred=True, steps=2,
                  seed=5, slots=[0] * 3 + list(range(4, 33)))
    got = [b for _, b in bench.plan_bytes(wl, "correction")]
    assert got == _bytes_by_loops(wl, tok=2306, rec=1024)
    wl1 = W.generate("tiny")
    assert [b for _, b in bench.plan_bytes(wl1, "correction")] == _bytes_by_loops(
        wl1, tok=2306, rec=1024)


def test_clock_summary_filters_the_timed_window():
    cs = bench.ClockSampler.__new__(bench.ClockSampler)
    cs.window = (100.0, 101.0)

    def row(sm, reason="Not Active", cap="Not Active"):
        return ["2026/01/01 00:00:00.000", str(sm), "2070", "900.0", "0x0", reason,
                "Not Active", "Not Active", cap]

    cs.samples = [(99.0, row(1000)), (100.2, row(2070)), (100.6, row(2040, cap="Active")),
                  (103.0, row(500, reason="Active"))]
    s = cs.summary()
    assert s["samples"] == 2 and s["sm_mhz"] == np.median([2070, 2040])
    assert s["reasons"] == ["sw_power_cap"]
    cs.samples = [(90.0, row(1800)), (100.5 + 5.0, row(1900))]
    s = cs.summary()                        # nothing inside: nearest sample
    assert s["samples"] == 1 and s["sm_mhz"] == 1900


_NCU_HEADER = ('"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream",'
               '"Block Size","Grid Size","Device","CC","Section Name","Metric Name",'
               '"Metric Unit","Metric Value"')


def _ncu_csv(path, launches):
    """An ncu --csv metrics log (one row per launch and metric)."""
    rows = ["==PROF== Connected to process 1 (python3)", _NCU_HEADER]
    for i, (kernel, metrics) in enumerate(launches):
        for name, unit, value in metrics:
            rows.append(f'"{i}","1","python3","host","{kernel}","1","7","(384, 1, 1)",'
                        f'"(152, 1, 1)","0","10.3","Command line profiler metrics","{name}",'
                        f'"{unit}","{value}"')
    path.write_text("\n".join(rows) + "\n")


def _fake_sources(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "profiles").mkdir()
    csrc = tmp_path / "linear_attention_speculative_kda_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "kda_kernels.cu").write_text("kernel v1")
    (csrc / "kda_conv.cu").write_text("conv v1")
    return csrc


def test_traffic_is_written_from_ncu_and_read_back(tmp_path, monkeypatch):
    csrc = _fake_sources(tmp_path, monkeypatch)
    kern = "void kda::step_kernel<(kda::Mode)0, false, false, false>(kda::Params, int, int)"
    csv_path = tmp_path / "dram.csv"
    _ncu_csv(csv_path, [
        (kern, [("dram__bytes_read.sum", "byte", "1,143,000,000"),
                ("dram__bytes_write.sum", "byte", "66,100,000"),
                ("gpu__time_duration.sum", "ns", "245000")]),
        (kern.replace(")0", ")1"), [("dram__bytes_read.sum", "Mbyte", "898.6"),
                                     ("dram__bytes_write.sum", "Gbyte", "0.8098"),
                                     ("gpu__time_duration.sum", "usecond", "296.9")])])
    wl = W.generate("tiny", pool=False)
    assert bench.launch_names(wl) == ["verify", "commit"]
    path = bench.write_traffic(str(csv_path), "w", bench.launch_names(wl), "ncu ... bench.py")
    data = json.loads(open(path).read())
    assert data["command"] == "ncu ... bench.py"
    assert data["launches"]["verify"]["traffic"] == 1143000000 + 66100000
    assert data["launches"]["commit"]["traffic"] == 898.6e6 + 0.8098e9
    assert data["launches"]["commit"]["duration_ns"] == 296900.0
    traffic, src = bench.profiled_traffic("verify", "w")
    assert traffic == 1209100000.0 and "profiles/ncu_w.json" in src
    assert bench.profiled_traffic("flush", "w")[0] is None
    (csrc / "kda_conv.cu").write_text("conv v2")   # not the step kernel's source
    assert bench.profiled_traffic("verify", "w")[0] == 1209100000.0
    (csrc / "kda_kernels.cu").write_text("kernel  v1 // a comment\n/* another */")
    assert bench.profiled_traffic("verify", "w")[0] == 1209100000.0   # comments and layout only
    (csrc / "kda_kernels.cu").write_text("kernel v2")
    traffic, src = bench.profiled_traffic("verify", "w")
    assert traffic is None and "other kernel sources" in src


def test_traffic_writer_refuses_a_partial_step(tmp_path, monkeypatch):
    _fake_sources(tmp_path, monkeypatch)
    csv_path = tmp_path / "dram.csv"
    _ncu_csv(csv_path, [("void kda::step_kernel<>(kda::Params, int, int)",
                         [("dram__bytes_read.sum", "byte", "1"),
                          ("dram__bytes_write.sum", "byte", "2")])])
    with pytest.raises(ValueError, match="one step has 4"):
        bench.write_traffic(str(csv_path), "d", bench.launch_names(W.generate(
            "deferred2", pool=False)), "")
    _ncu_csv(csv_path, [("at::FillFunctor", [("dram__bytes_read.sum", "byte", "1"),
                                             ("dram__bytes_write.sum", "byte", "2")])] * 2)
    with pytest.raises(ValueError, match="not the step kernel"):
        bench.write_traffic(str(csv_path), "t", ["verify", "commit"], "")


def test_code_text_strips_comments():
    src = "a = 1; // one\n/* two\n lines */ b  =\t2;"
    assert bench.code_text(src) == "a = 1; b = 2;"


def test_conv_compact_bytes_counts_rows_that_move():
    wl = W.custom(B=6, H=2, Q=4, lens=[4, 0, 3, 4, 2, 4], S=10, seed=8,
                  slots=[1, 2, 3, 0, 5, 6])
    # moved: rows 0 (n 2) and 4 (n clamped to 2); row 5 (n 1) leaves its
    # windows where they are
    acc = [2, 3, 0, 4, 9, 1]
    assert bench.conv_compact_bytes(wl, 768, 3, 2, acc) == 2 * 2 * 768 * 3 * 2


def test_align_commit_bytes_by_rows():
    wl = W.custom(B=4, H=2, Q=4, lens=[4, 4, 2, 4], S=10, seed=9, slots=[1, 2, 0, 3])
    acc = [3, 4, 2, 0]            # row 2 is null, row 3 commits nothing
    nc = [14, 0, 0, 0]            # row 0 reaches the boundary at 16 after 2 of 3 tokens
    per_head = (65536 + 3 * 770 + 2 * 65536) + (65536 + 4 * 770 + 65536)
    assert bench.align_commit_bytes(wl, None, nc, 16, acc) == 2 * per_head


def test_l2_note_is_truthful():
    assert bench.l2_note(2 * 10**9).startswith("inputs larger than L2 (state pool")
    note = bench.l2_note(2 * 2**20)
    assert note.startswith("inputs larger than L2: steps rotate over 247 copies")


def test_pool_copies_exceed_four_l2():
    for pool in (2 * 2**20, 201 * 10**6, 335 * 10**6, 600 * 10**6, 2 * 10**9):
        n = bench.pool_copies(pool)
        assert n * pool >= 4 * bench.L2_BYTES
        assert n == 1 or (n - 1) * pool < 4 * bench.L2_BYTES   # no more than needed
    assert bench.pool_copies(201 * 10**6) == 3 and bench.pool_copies(2 * 10**9) == 1


def test_reference_arm_prints_the_contract_line():
    """The reference arm (the oracle on the host cores) runs without a GPU and
    prints one JSON line with the fields the benchmark contract names."""
    import json
    import subprocess
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--config", "tiny", "--steps", "2", "--warmup", "1"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    line = json.loads(res.stdout.strip().splitlines()[-1])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["config"]["workload"] == "tiny"


def test_cpu_baseline_reports_three_legs():
    """The CPU baseline times the fp64 oracle on all cores (its value), the
    float build of the same C code on all cores and the oracle on one core."""
    line = bench.cpu_baseline(W.generate("tiny"), 0.2)
    legs = line["legs"]
    assert [(leg["arithmetic"], leg["cores"]) for leg in legs] == [
        ("fp64", line["cores"]), ("fp32", line["cores"]), ("fp64", 1)]
    assert line["kind"] == "oracle" and line["value"] == legs[0]["value"]
    assert all(leg["value"] > 0 for leg in legs)


def test_record_blocks_bytes_by_recorded_rows():
    # 3 rows read their slot (12 bytes); 2 have one and move 16 bytes each
    assert bench.record_blocks_bytes([4, -1, 0]) == 3 * 4 + 2 * 16
    assert bench.record_blocks_bytes([]) == 0


def test_plan_fp32_ops_by_hand():
    # eager workload: rows of T = 4, 0, 2 (the middle one a null row), H = 2
    wl = W.custom(B=3, H=2, Q=4, lens=[4, 3, 2], S=6, seed=3, slots=[1, 0, 2])
    wl.steps[0].num_accepted[:] = torch.tensor([3, 4, 9])
    ops = dict(bench.plan_fp32_ops(wl))
    E = 128 * 128
    assert ops["verify"] == (4 + 2) * 2 * 4 * E          # live rows' tokens x H x 4
    assert ops["commit"] == (3 + 2) * 2 * 3 * E          # n = 3 and min(9, 2) = 2
    assert dict(bench.plan_fp32_ops(wl, "correction"))["commit"] == (3 + 2) * 2 * 2 * E


def test_plan_fp32_ops_deferred_steps():
    wl = W.custom(B=4, H=1, Q=4, lens=[4, 4, 4, 4], S=6, R=4, deferred=True, steps=2, seed=5)
    wl.steps[0].num_accepted[:] = torch.tensor([2, 3, 0, 4])
    wl.steps[0].eager[:] = torch.tensor([1, 0, 0, 0], dtype=torch.uint8)
    wl.steps[1].num_accepted[:] = torch.tensor([1, 1, 1, 1])
    ops = dict(bench.plan_fp32_ops(wl))
    E = 128 * 128
    assert ops["verify"] == 16 * 4 * E
    assert ops["commit_deferred"] == 2 * 3 * E            # the eager row replays 2
    assert ops["verify_fused"] == 16 * 4 * E + (3 + 4) * 3 * E   # folds 3 and 4 pending
    assert ops["commit"] == 4 * 3 * E


def test_flush_bytes_counts_pending_rows():
    wl = W.custom(B=4, H=2, Q=4, lens=[4, 4, 2, 4], S=6, R=4, deferred=True, steps=2, seed=5,
                  slots=[1, 2, 3, 0])
    wl.steps[0].num_accepted[:] = torch.tensor([2, 3, 9, 4])
    wl.steps[0].eager[:] = torch.tensor([1, 0, 0, 0], dtype=torch.uint8)
    # pending: row 1 (3) and row 2 (min(9, 2) = 2); row 0 is eager, row 3 a null row
    want = 2 * ((131072 + 3 * bench.RECORD_BYTES) + (131072 + 2 * bench.RECORD_BYTES))
    assert bench.flush_bytes(wl) == want


def test_conv_align_bytes_against_the_oracle_moves():
    # the rows the oracle's align conv compaction moves, and how many windows
    import numpy as np
    from oracle import kda_oracle as O
    wl = W.custom(B=6, H=1, Q=4, lens=[4, 4, 2, 3, 4, 1], S=7, seed=2, slots=[1, 2, 0, 3, 4, 5])
    acc = [3, 4, 2, 1, 0, 1]
    # row 0 passes the boundary at 16 (two blocks); row 3 ends on it, so its
    # boundary block is its final block (one); rows 1 and 5 stay in one block
    num_computed = [14, 3, 5, 15, 0, 16]
    C, width, Q = 8, 6, 4
    hist = width - Q + 1
    S = 1 + 6 + 6 * 2
    table = (7 + np.arange(12)).reshape(6, 2)
    conv = np.arange(S * C * width, dtype=np.float64).reshape(S, C, width)
    new, issues = O.conv_compact_align(conv, wl.cu_seqlens.numpy(), wl.state_indices.numpy(),
                                       np.array(acc), Q, table, np.array(num_computed), 16)
    assert issues == []
    # every window the oracle wrote is a block whose columns [0, hist) changed
    written = sum(1 for s in range(S) if not np.array_equal(new[s, :, :hist], conv[s, :, :hist]))
    got = bench.conv_align_bytes(wl, num_computed, 16, acc, C, hist, 2)
    assert got == written * 2 * C * hist * 2
