"""Benchmark of KDA speculative verify + commit on GB300.

One step is one pass of the whole hot path over one batch.  For the default
workload (deferred2: B=1024 requests, H=16 heads, Q=4, deferred commit over
two chained decode steps) a step is the four launches
    verify(step 1) -> deferred commit(step 1, 10% eager)
    -> verify(step 2, folding the pending replays) -> commit(step 2, all eager)
so every step starts and ends with no pending replay.  Other workloads run
verify -> eager commit.  The metric is (request*head)-steps per second: each
decode step of each (request, head) pair counts once.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on a
bounded sample of the same workload instead (the reference arm).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from linear_attention_speculative_kda_gb300 import workloads as W  # noqa: E402

METRIC = "verify+commit (request*head)-steps/s"
UNIT = "(request*head)-steps/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0

STATE_BYTES = 128 * 128 * 4          # one fp32 state tile
TOKEN_BYTES = 2052                   # q, k, v, g_raw, beta read + out, records written
RECORD_BYTES = 770                   # raw k, v, g_raw, beta read back by a replay
# correction records: fp32 delta + bf16 k + bf16 g_raw (1024 bytes) per token
CORR_TOKEN_BYTES = 1024 + 2 + 256 + 1024
CORR_RECORD_BYTES = 1024


def format_bytes(record_format: str):
    """(bytes a verify moves per new token, bytes a replay reads per record)."""
    if record_format == "correction":
        return CORR_TOKEN_BYTES, CORR_RECORD_BYTES
    return TOKEN_BYTES, RECORD_BYTES


# ---------------------------------------------------------------- helpers --

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def max_over_ranks(x: float, world: int, device) -> float:
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device) -> float:
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


def shard_seed(base_seed: int, rank: int) -> int:
    """Weak scaling: every rank draws its own batch of the same shape."""
    return base_seed + 1000 * rank


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            data = json.load(fh)
    except (OSError, ValueError):
        return None
    return data


def hbm_peak():
    data = measured_peaks()
    if data:
        for key in ("hbm_gbs", "hbm_GBs", "hbm"):
            if key in data and isinstance(data[key], (int, float)):
                return float(data[key]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


# the sources of the verify / commit kernel (the conv kernel has its own file)
STEP_SOURCES = ("kda_align.cuh", "kda_async.cuh", "kda_device.cuh", "kda_kernels.cu", "kda_tc.cuh")


_COMMENT = re.compile(r"//[^\n]*|/\*.*?\*/", re.S)


def code_text(source: str) -> str:
    """C/CUDA source without its comments and with its whitespace collapsed
    (the step sources hold no string literal with comment markers), so that
    a comment edit does not change the hash below."""
    return " ".join(_COMMENT.sub(" ", source).split())


def kernel_source_hash() -> str:
    """Hash of the verify / commit kernel's code (comments and layout
    aside): a profile taken on other code no longer describes the kernel."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "linear_attention_speculative_kda_gb300", "csrc")
    for name in STEP_SOURCES:
        path = os.path.join(csrc, name)
        if not os.path.exists(path):
            continue
        with open(path, encoding="utf-8") as fh:
            h.update(name.encode())
            h.update(code_text(fh.read()).encode())
    return h.hexdigest()[:16]


def traffic_path(workload: str) -> str:
    return os.path.join(ROOT, "profiles", f"ncu_{workload}.json")


def profiled_traffic(launch: str, workload: str):
    """(DRAM bytes of one launch, where they came from): the ncu counters
    dram__bytes_read.sum + dram__bytes_write.sum that ``--ncu-traffic``
    wrote to profiles/ncu_<workload>.json from a capture of the same
    launch, if that capture was taken on the current kernel sources; else
    (None, why not)."""
    path = traffic_path(workload)
    rel = os.path.relpath(path, ROOT)
    try:
        with open(path) as fh:
            data = json.load(fh)
    except (OSError, ValueError):
        return None, f"no capture ({rel} missing)"
    if data.get("source_hash") != kernel_source_hash():
        return None, f"{rel} was captured on other kernel sources"
    entry = data.get("launches", {}).get(launch)
    if not entry:
        return None, f"{rel} holds no launch named {launch}"
    return (float(entry["traffic"]),
            f"{rel}: ncu dram__bytes_read.sum + dram__bytes_write.sum of launch {launch}")


def _ncu_value(value: str, unit: str) -> float:
    scale = {"byte": 1.0, "kbyte": 1e3, "mbyte": 1e6, "gbyte": 1e9, "tbyte": 1e12,
             "nsecond": 1.0, "usecond": 1e3, "msecond": 1e6, "second": 1e9,
             "ns": 1.0, "us": 1e3, "ms": 1e6, "s": 1e9}
    factor = scale.get(unit.strip().lower())
    if factor is None:
        raise ValueError(f"unexpected ncu unit {unit!r}")
    return float(value.replace(",", "")) * factor


def read_ncu_csv(path: str):
    """Launches of an ncu ``--csv`` metrics log, in capture order: a list of
    (kernel name, {metric: value in bytes or nanoseconds})."""
    import csv
    with open(path, newline="") as fh:
        lines = fh.read().splitlines()
    start = next(i for i, ln in enumerate(lines) if ln.startswith('"ID"'))
    launches = {}
    for row in csv.DictReader(lines[start:]):
        if not row.get("ID"):
            continue
        name, metrics = launches.setdefault(row["ID"], (row["Kernel Name"], {}))
        metrics[row["Metric Name"]] = _ncu_value(row["Metric Value"], row["Metric Unit"])
    return [launches[k] for k in sorted(launches, key=int)]


def write_traffic(csv_path: str, workload: str, names, command: str) -> str:
    """Write profiles/ncu_<workload>.json from an ncu capture of exactly the
    launches of one step (``names``, in launch order)."""
    launches = read_ncu_csv(csv_path)
    if len(launches) != len(names):
        raise ValueError(f"the capture holds {len(launches)} launches, one step has "
                         f"{len(names)} ({', '.join(names)})")
    out = {"workload": workload, "source_hash": kernel_source_hash(), "command": command,
           "metric": "dram__bytes_read.sum + dram__bytes_write.sum (bytes per launch)",
           "launches": {}}
    for name, (kernel, m) in zip(names, launches):
        if "step_kernel" not in kernel:
            raise ValueError(f"launch {name} is {kernel}, not the step kernel")
        rd, wr = m["dram__bytes_read.sum"], m["dram__bytes_write.sum"]
        out["launches"][name] = {"kernel": kernel, "dram_bytes_read": rd,
                                 "dram_bytes_write": wr, "traffic": rd + wr,
                                 "duration_ns": m.get("gpu__time_duration.sum")}
    path = traffic_path(workload)
    with open(path, "w") as fh:
        json.dump(out, fh, indent=1)
        fh.write("\n")
    return path


def launch_names(wl: W.Workload):
    """Names of one step's launches (the capture order of a step)."""
    if wl.spec.deferred:
        return ["verify", "commit_deferred", "verify_fused", "commit"]
    return ["verify", "commit"]


class ClockSampler:
    """nvidia-smi clock / throttle sampling around the timed region.

    Started before the warm-up so the sampler is running when the timed
    region begins; ``mark(start, stop)`` gives the host wall-clock bounds of
    the timed region and ``summary()`` keeps the samples taken inside it
    (or the nearest one when the region is shorter than the 200 ms period).
    """

    QUERY = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.gpu_id = self._smi_id(device_index)
        self.proc = None
        self.samples: list[tuple[float, list[str]]] = []
        self.thread = None
        self.window = None

    @staticmethod
    def _smi_id(device_index: int) -> str:
        """nvidia-smi id of the torch device (its UUID; the visible-devices
        list maps torch indices to physical ones)."""
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            if uuid:
                return uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            pass
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        return ids[device_index] if device_index < len(ids) else str(device_index)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_id}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [p.strip() for p in line.split(",")]))

    def mark(self, start: float, stop: float):
        self.window = (start, stop)

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread is not None:
                self.thread.join(timeout=2)

    def summary(self):
        rows = [(t, p) for t, p in self.samples if len(p) >= 9]
        if self.window and rows:
            lo, hi = self.window
            inside = [(t, p) for t, p in rows if lo <= t <= hi + 0.2]
            if not inside:
                mid = 0.5 * (lo + hi)
                inside = [min(rows, key=lambda r: abs(r[0] - mid))]
            rows = inside
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, parts in rows:
            try:
                sms.append(float(parts[1]))
                maxes.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes),
                "reasons": sorted(reasons), "samples": len(sms)}


# ------------------------------------------------------- algorithmic bytes --

def plan_bytes(wl: W.Workload, record_format: str = "raw"):
    """Algorithmic bytes of each launch of one step, from the drawn lengths,
    accepted counts, eager masks and the pending replays they imply."""
    tok_b, rec_b = format_bytes(record_format)
    sp = wl.spec
    H = sp.H
    lens = wl.lens.numpy().astype(np.int64)
    slots = wl.state_indices.numpy()
    live = slots > 0

    def commit_n(acc):
        return np.minimum(np.maximum(acc, 0), np.minimum(lens, sp.Q))

    launches = []
    if not sp.deferred:
        n = commit_n(wl.steps[0].num_accepted.numpy().astype(np.int64))
        vb = np.where(live & (lens > 0), STATE_BYTES + lens * tok_b, 0).sum() * H
        cb = np.where(live & (n > 0), 2 * STATE_BYTES + n * rec_b, 0).sum() * H
        launches = [("verify", float(vb)), ("commit", float(cb))]
        return launches
    n1 = commit_n(wl.steps[0].num_accepted.numpy().astype(np.int64))
    eager1 = wl.steps[0].eager.numpy().astype(bool)
    n2 = commit_n(wl.steps[1].num_accepted.numpy().astype(np.int64))
    valid1 = live & (n1 > 0)
    v1 = np.where(live & (lens > 0), STATE_BYTES + lens * tok_b, 0).sum() * H
    c1 = np.where(valid1 & eager1, 2 * STATE_BYTES + n1 * rec_b, 0).sum() * H
    pend = np.where(valid1 & ~eager1, n1, 0)
    v2 = np.where(live & ((lens > 0) | (pend > 0)),
                  STATE_BYTES + lens * tok_b
                  + np.where(pend > 0, STATE_BYTES + pend * rec_b, 0), 0).sum() * H
    c2 = np.where(live & (n2 > 0), 2 * STATE_BYTES + n2 * rec_b, 0).sum() * H
    return [("verify", float(v1)), ("commit_deferred", float(c1)),
            ("verify_fused", float(v2)), ("commit", float(c2))]


STATE_ELEMS = 128 * 128
FP32_LANES_PER_SM = 128  # 4 SMSPs x 32 FP32 lanes


def plan_fp32_ops(wl: W.Workload, record_format: str = "raw"):
    """Algorithmic FP32 operations (a multiply or a fused multiply-add each
    counts one) of each launch of one step, from the same drawn counts as
    plan_bytes: per state element, 4 per verified token (the decay, u = S k^,
    the rank-one update and o = S q^) and 3 per replayed token (no output;
    2 with correction records, which skip u)."""
    rep_ops = 2 if record_format == "correction" else 3
    sp = wl.spec
    H = sp.H
    lens = wl.lens.numpy().astype(np.int64)
    live = wl.state_indices.numpy() > 0

    def commit_n(acc):
        return np.minimum(np.maximum(acc, 0), np.minimum(lens, sp.Q))

    def ops(tokens, per):
        return float(np.where(live, tokens, 0).sum() * H * per * STATE_ELEMS)

    v1 = ops(lens, 4)
    if not sp.deferred:
        n = commit_n(wl.steps[0].num_accepted.numpy().astype(np.int64))
        return [("verify", v1), ("commit", ops(n, rep_ops))]
    n1 = commit_n(wl.steps[0].num_accepted.numpy().astype(np.int64))
    eager1 = wl.steps[0].eager.numpy().astype(bool)
    n2 = commit_n(wl.steps[1].num_accepted.numpy().astype(np.int64))
    pend = np.where(live & (n1 > 0) & ~eager1, n1, 0)
    return [("verify", v1), ("commit_deferred", ops(np.where(eager1, n1, 0), rep_ops)),
            ("verify_fused", v1 + ops(pend, rep_ops)), ("commit", ops(n2, rep_ops))]


def fp32_peak(device, clock_summary):
    """FP32 FMA-pipe peak in T ops/s from the unit counts: SMs x 128 lanes x
    the SM clock sampled during the run (else the part's 2,070 MHz maximum)."""
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    mhz = clock_summary.get("sm_mhz") or 2070.0
    src = ("sampled SM clock" if clock_summary.get("sm_mhz") else "maximum SM clock")
    return sms * FP32_LANES_PER_SM * mhz * 1e6 / 1e12, (
        f"{sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x {mhz:.0f} MHz ({src})")


def units_per_step(wl: W.Workload) -> int:
    return wl.spec.B * wl.spec.H * wl.spec.steps


# ------------------------------------------------------------- GPU engine --

class Engine:
    """Device-resident buffers of one workload and the step's launches."""

    def __init__(self, wl: W.Workload, device, record_format: str = "raw"):
        from linear_attention_speculative_kda_gb300 import api
        self.api = api
        self.wl = wl
        sp = wl.spec
        d = device
        self.dev = d
        self.A_log = wl.A_log.to(d)
        self.g_bias = wl.g_bias.to(d)
        # consecutive steps run on different copies of the state pool, enough
        # of them that a step finds none of its checkpoints in L2
        self.pools = [wl.pool.to(d)]
        for _ in range(pool_copies(wl.pool.numel() * 4) - 1):
            self.pools.append(self.pools[0].clone())
        self.pool = self.pools[0]
        self.turn = 0
        self.cu = wl.cu_seqlens.to(d)
        self.slots = wl.state_indices.to(d)
        self.rr = None if wl.record_rows is None else wl.record_rows.to(d)
        self.records = api.allocate_records(sp.H, sp.Q, sp.record_slots, d,
                                            record_format=record_format)
        self.pending = torch.zeros(sp.record_slots, dtype=torch.int32, device=d)
        self.err = torch.zeros(1, dtype=torch.int32, device=d)
        self.all_eager = torch.ones(sp.B, dtype=torch.uint8, device=d)
        self.steps = self.new_input_set()
        self.kw = dict(window=sp.Q, record_slots=sp.record_slots,
                       lower_bound=sp.lower_bound if sp.bounded else None,
                       record_format=record_format)

    def new_input_set(self):
        """Device copies of every decode step's inputs, plus output buffers."""
        sp, d = self.wl.spec, self.dev
        T = self.wl.total_tokens
        steps = []
        for st in self.wl.steps:
            steps.append(dict(
                qkv=st.qkv.to(d), beta_buf=st.beta_buf.to(d), g_raw=st.g_raw.to(d),
                num_accepted=st.num_accepted.to(d),
                eager=None if st.eager is None else st.eager.to(d),
                out=torch.empty((T, sp.H, sp.D), dtype=torch.bfloat16, device=d)))
        return steps

    def _verify(self, s, pending, pool):
        H = self.wl.spec.H
        self.api.kda_verify(s["qkv"][:, 0], s["qkv"][:, 1], s["qkv"][:, 2], s["g_raw"],
                            s["beta_buf"][:, :H], self.A_log, self.g_bias, pool, self.cu,
                            self.slots, self.records, s["out"], record_rows=self.rr,
                            pending=self.pending if pending else None, error_word=self.err,
                            **self.kw)

    def _commit(self, s, deferred, eager, pool):
        self.api.kda_commit(self.A_log, self.g_bias, pool, self.cu, self.slots,
                            s["num_accepted"], self.records, record_rows=self.rr,
                            pending=self.pending if deferred else None,
                            eager=eager if deferred else None, error_word=self.err, **self.kw)

    def launches(self, steps=None, pool=None):
        """The step as a list of (name, callable), on input set `steps` and
        state pool `pool` (by default the first copy)."""
        steps = self.steps if steps is None else steps
        pool = self.pool if pool is None else pool
        if not self.wl.spec.deferred:
            s = steps[0]
            return [("verify", lambda: self._verify(s, False, pool)),
                    ("commit", lambda: self._commit(s, False, None, pool))]
        s1, s2 = steps
        # the step ends with every row committed (pending all 0), so the next
        # step may run on another copy of the pool
        return [("verify", lambda: self._verify(s1, True, pool)),
                ("commit_deferred", lambda: self._commit(s1, True, s1["eager"], pool)),
                ("verify_fused", lambda: self._verify(s2, True, pool)),
                ("commit", lambda: self._commit(s2, True, self.all_eager, pool))]

    def run_step(self, events=None, steps=None):
        pool = self.pools[self.turn % len(self.pools)]
        self.turn += 1
        for i, (_, fn) in enumerate(self.launches(steps, pool)):
            if events is not None:
                events[i][0].record()
            fn()
            if events is not None:
                events[i][1].record()


class HostIO:
    """End-to-end steps through the public API with host buffers: every step
    copies its inputs from pinned host memory to the device, runs the
    launches, and copies its outputs back to pinned host memory.  Two device
    input sets and three streams (copy-in, compute, copy-out) let step j+1's
    inputs travel and step j-1's outputs return while step j computes, as a
    serving loop would.  The dependencies, per input set s: its inputs are
    overwritten once the compute that read them is done; its outputs once
    they have been copied out."""

    KEYS = ("qkv", "beta_buf", "g_raw", "num_accepted", "eager")

    def __init__(self, eng: Engine):
        self.eng = eng
        self.sets = [eng.steps, eng.new_input_set()]
        self.h_in = []
        for st in eng.steps:
            self.h_in.append({k: st[k].cpu().pin_memory() for k in self.KEYS
                              if st[k] is not None})
        self.h_out = [[torch.empty(st["out"].shape, dtype=st["out"].dtype).pin_memory()
                       for st in eng.steps] for _ in range(2)]
        self.h2d = sum(t.numel() * t.element_size() for ins in self.h_in for t in ins.values())
        self.d2h = sum(t.numel() * t.element_size() for t in self.h_out[0])
        self.copy_in = torch.cuda.Stream(eng.dev)
        self.copy_out = torch.cuda.Stream(eng.dev)
        self._reset()

    def _reset(self):
        self.done = [None, None]     # compute on set s finished (its inputs are free)
        self.freed = [None, None]    # set s's outputs copied out (its out buffers are free)
        self.arrived = [None, None]  # set s's inputs in place

    def _copy_in(self, s: int):
        with torch.cuda.stream(self.copy_in):
            if self.done[s] is not None:
                self.copy_in.wait_event(self.done[s])
            for st, ins in zip(self.sets[s], self.h_in):
                for k, t in ins.items():
                    st[k].copy_(t, non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(self.copy_in)
            self.arrived[s] = ev

    def _compute_and_copy_out(self, s: int, comp):
        if self.arrived[s] is not None:
            comp.wait_event(self.arrived[s])
        if self.freed[s] is not None:
            comp.wait_event(self.freed[s])
        self.eng.run_step(steps=self.sets[s])
        done = torch.cuda.Event()
        done.record(comp)
        self.done[s] = done
        with torch.cuda.stream(self.copy_out):
            self.copy_out.wait_event(done)
            for st, out in zip(self.sets[s], self.h_out[s]):
                out.copy_(st["out"], non_blocking=True)
            freed = torch.cuda.Event()
            freed.record(self.copy_out)
            self.freed[s] = freed

    def _issue(self, k_steps: int, first_filled: bool, fill_next: bool):
        """Steps 0 .. k_steps - 1 on input sets 0, 1, 0, ...; the copy of step
        j + 1's inputs is issued before step j computes.  first_filled: set 0
        already holds step 0's inputs; fill_next: the last step also fills
        set 0 for a following step 0."""
        comp = torch.cuda.current_stream(self.eng.dev)
        go = torch.cuda.Event()
        go.record(comp)
        self.copy_in.wait_event(go)
        self.copy_out.wait_event(go)
        if not first_filled:
            self._copy_in(0)
        for j in range(k_steps):
            s = j & 1
            if j + 1 < k_steps:
                self._copy_in(s ^ 1)
            elif fill_next:
                self._copy_in(0)
            self._compute_and_copy_out(s, comp)
        comp.wait_stream(self.copy_in)
        comp.wait_stream(self.copy_out)
        self._reset()

    def run(self, k_steps: int):
        """Issue k_steps steps from the host, call by call."""
        self._issue(k_steps, first_filled=False, fill_next=False)

    def graph_steps(self) -> int:
        """Steps in one captured graph: a whole number of turns of the state
        pools (so that replays keep their rotation) and of the two input
        sets, at least 8."""
        n = math.lcm(2, len(self.eng.pools))
        return n * max(1, -(-8 // n))

    def capture(self):
        """The same steps captured once into a CUDA graph of graph_steps()
        steps, for replay: every step's public API calls, host-to-device
        input copies and device-to-host output copies.  A replay starts with
        set 0 filled (fill_first before the first one) and ends by filling
        it for the next, so that the input copies overlap compute across
        replays too."""
        self._reset()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            self._issue(self.graph_steps(), first_filled=True, fill_next=True)
        return graph

    def fill_first(self):
        """Input set 0 for the first replay, on the current stream."""
        for st, ins in zip(self.sets[0], self.h_in):
            for k, t in ins.items():
                st[k].copy_(t, non_blocking=True)


# -------------------------------------------------------------- CPU side --

def oracle_sample_run(wl: W.Workload, rows, threads: int, record_format: str = "raw"):
    """The oracle on a sample of rows of the workload's whole step; returns
    (units processed, seconds)."""
    from oracle import kda_oracle as O

    def f64(t):
        return t.to(torch.float64).numpy()

    sp = wl.spec
    layer = O.Layer(sp.H, sp.D, sp.Q, f64(wl.A_log), f64(wl.g_bias).reshape(sp.H, sp.D),
                    sp.bounded, sp.lower_bound if sp.bounded else 0.0, wl.scale)
    steps = [O.Step(f64(st.q), f64(st.k), f64(st.v), f64(st.g_raw), f64(st.beta_raw),
                    wl.cu_seqlens.numpy(), wl.state_indices.numpy(),
                    None if wl.record_rows is None else wl.record_rows.numpy())
             for st in wl.steps]
    cache = O.Cache(wl.pool.numpy(), sp.record_slots, record_format=record_format)
    t0 = time.perf_counter()
    if not sp.deferred:
        O.verify(layer, cache, steps[0], rows=rows, threads=threads)
        O.commit(layer, cache, steps[0], wl.steps[0].num_accepted.numpy(), rows=rows,
                 threads=threads)
    else:
        st1, st2 = wl.steps
        O.verify(layer, cache, steps[0], pending=True, rows=rows, threads=threads)
        O.commit(layer, cache, steps[0], st1.num_accepted.numpy(), deferred=True,
                 eager=st1.eager.numpy(), rows=rows, threads=threads)
        O.verify(layer, cache, steps[1], pending=True, rows=rows, threads=threads)
        O.commit(layer, cache, steps[1], st2.num_accepted.numpy(), deferred=True,
                 eager=np.ones(sp.B, np.uint8), rows=rows, threads=threads)
    dt = time.perf_counter() - t0
    return len(rows) * sp.H * sp.steps, dt


def time_oracle(wl: W.Workload, budget_s: float, threads: int, record_format: str = "raw",
                arithmetic: str = "fp64"):
    """Time the oracle (or its float build) on growing samples of rows until
    ``budget_s`` seconds of CPU work have been measured (or the whole batch
    is done).  Returns (units per second, rows done, seconds)."""
    from oracle import kda_oracle as O
    rng = np.random.default_rng(123)
    order = rng.permutation(wl.spec.B).tolist()
    units = 0
    secs = 0.0
    done = 0
    chunk = max(1, threads)
    with O.arithmetic(arithmetic):
        while done < len(order) and secs < budget_s:
            rows = order[done:done + chunk]
            u, dt = oracle_sample_run(wl, rows, threads, record_format)
            units += u
            secs += dt
            done += len(rows)
            chunk = min(len(order) - done, chunk * 2) if done < len(order) else 0
            if chunk <= 0:
                break
    return (units / secs if secs > 0 else None), done, secs


def cpu_baseline(wl: W.Workload, budget_s: float, record_format: str = "raw"):
    """The CPU baseline: the fp64 oracle on all host cores (the reported
    value), beside the float build of the same C code on all cores and the
    fp64 oracle on one core, each on a bounded sample of the workload."""
    threads = max(1, os.cpu_count() or 1)
    legs = []
    for arith, nthreads, budget in (("fp64", threads, budget_s),
                                    ("fp32", threads, budget_s / 2),
                                    ("fp64", 1, budget_s / 2)):
        value, done, secs = time_oracle(wl, budget, nthreads, record_format, arith)
        legs.append({"arithmetic": arith, "cores": nthreads, "value": value,
                     "sample": f"{done} of {wl.spec.B} rows x {wl.spec.H} heads x "
                               f"{wl.spec.steps} decode step(s), {secs:.1f} s"})
    main = legs[0]
    return {"value": main["value"], "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{main['sample']} of workload {wl.spec.name}, fp64 C oracle, "
                      f"{threads} threads",
            "legs": legs}


# ------------------------------------------------------------------- arms --

def workload_config(wl: W.Workload, world: int, record_format: str = "raw"):
    sp = wl.spec
    return {"workload": sp.name, "records": record_format,
            "requests": sp.B, "heads": sp.H, "head_dim": sp.D,
            "window": sp.Q, "pool_slots": sp.S, "record_slots": sp.record_slots,
            "gate": f"bounded lb={sp.lower_bound}" if sp.bounded else "softplus",
            "decode_steps_per_step": sp.steps, "ranks": world,
            "tokens_per_decode_step": wl.total_tokens,
            "state": "f32", "activations": "bf16",
            "l2": l2_note(wl.pool.numel() * 4)}


L2_BYTES = 129 * 10**6   # GB300 L2
POOL_ROTATION_BYTES = 4 * L2_BYTES


def pool_copies(pool_bytes: int) -> int:
    """Copies of the state pool that consecutive steps rotate over: enough to
    hold 4x the L2 in all, so that a step's checkpoints (written by the step
    that used the same copy, several steps before) have left L2."""
    if pool_bytes <= 0:
        return 1
    return max(1, -(-POOL_ROTATION_BYTES // pool_bytes))


def l2_note(pool_bytes: int) -> str:
    n = pool_copies(pool_bytes)
    if n == 1:
        return "inputs larger than L2 (state pool %.2f GB)" % (pool_bytes / 1e9)
    return ("inputs larger than L2: steps rotate over %d copies of the %.3f GB state pool "
            "(%.2f GB in all)" % (n, pool_bytes / 1e9, n * pool_bytes / 1e9))


def conv_compact_bytes(wl: W.Workload, conv_dim: int, hist: int, elem_bytes: int, acc) -> int:
    """Algorithmic bytes of one conv compaction: every row that moves its
    windows (slot > 0, n > 1; with n = 1 each window is already at column 0)
    reads its window of conv_dim x history elements and writes it back at
    column 0."""
    lens = (wl.cu_seqlens[1:] - wl.cu_seqlens[:-1]).tolist()
    slots = wl.state_indices.tolist()
    rows = sum(1 for b in range(wl.spec.B)
               if slots[b] > 0 and min(max(int(acc[b]), 0), lens[b], wl.spec.Q) > 1)
    return 2 * rows * conv_dim * hist * elem_bytes


def time_launches(launch, iters: int, warmup: int):
    """Average device time (us) of ``launch(k)`` for k in range(iters),
    replayed from one CUDA graph so that the host's per-call cost does not
    show in short launches.  Returns (us, how)."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for k in range(warmup):
            launch(k)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for k in range(iters):
            launch(k)
    graph.replay()
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    graph.replay()
    stop.record()
    torch.cuda.synchronize()
    del graph
    return start.elapsed_time(stop) * 1e3 / iters, "cuda graph"


def measure_conv_compact(wl: W.Workload, device, iters: int, warmup: int, peak: float,
                         layout: str = "dim_first"):
    """The conv-state compaction of the workload's commit (bf16 pool
    [S, 3*H*D, history + Q - 1], channel-major or column-major), timed alone
    from a CUDA graph replay.  Three pool copies in rotation keep each
    launch's pool out of L2."""
    from linear_attention_speculative_kda_gb300 import api
    S, C, width = W.conv_shape(wl.spec)

    def on_device(t):  # keep the storage order of the host pool
        return t.to(device) if layout == "dim_first" else \
            t.transpose(1, 2).contiguous().to(device).transpose(1, 2)

    pools = [on_device(W.conv_state(S, C, width, seed=i, layout=layout)) for i in range(3)]
    i32 = dict(dtype=torch.int32, device=device)
    cu = wl.cu_seqlens.to(**i32)
    slots = wl.state_indices.to(**i32)
    acc = wl.steps[0].num_accepted.to(**i32)
    err = torch.zeros(1, **i32)

    def launch(k):
        api.kda_conv_compact(pools[k % 3], cu, slots, acc, window=wl.spec.Q, error_word=err)

    us, how = time_launches(launch, iters, warmup)
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())} in the conv compaction")
    b = conv_compact_bytes(wl, C, width - wl.spec.Q + 1, 2, wl.steps[0].num_accepted.tolist())
    del pools
    return {"shape": [S, C, width], "dtype": "bf16", "timing": how,
            "layout": "channel-major" if layout == "dim_first" else "column-major",
            "launches": iters, "avg_us": us, "bytes_per_launch": b,
            "gbs": b / (us / 1e6) / 1e9, "frac": b / (us / 1e6) / 1e9 / peak}


def flush_bytes(wl: W.Workload, record_format: str = "raw") -> int:
    """Algorithmic bytes of one flush after the first step's deferred commit:
    every (row, head) with a pending replay (slot > 0, n > 0, not eager)
    reads its checkpoint and its p records and writes the checkpoint."""
    _, rec_b = format_bytes(record_format)
    sp = wl.spec
    lens = wl.lens.numpy().astype(np.int64)
    live = wl.state_indices.numpy() > 0
    acc = wl.steps[0].num_accepted.numpy().astype(np.int64)
    n1 = np.minimum(np.maximum(acc, 0), np.minimum(lens, sp.Q))
    eager1 = wl.steps[0].eager.numpy().astype(bool)
    pend = np.where(live & (n1 > 0) & ~eager1, n1, 0)
    return int(np.where(pend > 0, 2 * STATE_BYTES + pend * rec_b, 0).sum() * sp.H)


def measure_flush(wl: W.Workload, device, iters: int, warmup: int, peak: float,
                  record_format: str = "raw"):
    """kda_flush after the first step's verify and deferred commit (the
    pending replays of every deferred row), timed alone from a CUDA graph
    replay.  Every launch folds the same pending counts, so each moves the
    same bytes."""
    eng = Engine(wl, device, record_format)
    fns = dict(eng.launches())
    fns["verify"]()
    fns["commit_deferred"]()

    def launch(_k):
        eng.api.kda_flush(eng.A_log, eng.g_bias, eng.pool, eng.slots, eng.records, eng.pending,
                          record_rows=eng.rr, error_word=eng.err, **eng.kw)

    us, how = time_launches(launch, iters, warmup)
    if int(eng.err.item()) != 0:
        raise RuntimeError(f"device error word {int(eng.err.item())} in the flush")
    b = flush_bytes(wl, record_format)
    del eng
    return {"timing": how, "launches": iters, "avg_us": us, "bytes_per_launch": b,
            "gbs": b / (us / 1e6) / 1e9, "frac": b / (us / 1e6) / 1e9 / peak}


def align_commit_bytes(wl: W.Workload, table, num_computed, block_size: int, acc) -> int:
    """Algorithmic bytes of one align-mode commit: every committing (row,
    head) reads its checkpoint and n records and writes the final block, plus
    the boundary block when the boundary comes before the last token."""
    lens = (wl.cu_seqlens[1:] - wl.cu_seqlens[:-1]).tolist()
    slots = wl.state_indices.tolist()
    total = 0
    for b in range(wl.spec.B):
        n = min(max(int(acc[b]), 0), lens[b], wl.spec.Q)
        if slots[b] <= 0 or n <= 0:
            continue
        c = int(num_computed[b])
        boundary = (c // block_size + 1) * block_size
        mid = c + n >= boundary and boundary - c < n
        total += 65536 + n * 770 + 65536 * (2 if mid else 1)
    return total * wl.spec.H


def record_blocks_bytes(idx_mapping) -> int:
    """Algorithmic bytes of one kda_record_state_blocks launch with one spec
    row per request: every row reads its request's running slot (4 bytes);
    a row with a slot also reads num_computed and num_sampled and writes the
    column and the accepted count (16 bytes)."""
    recorded = sum(1 for s in idx_mapping if int(s) >= 0)
    return 4 * len(idx_mapping) + 16 * recorded


def measure_record_state_blocks(wl: W.Workload, device, iters: int, warmup: int):
    """The align-mode bookkeeping after the commit on the workload's rows, timed
    alone from a CUDA graph replay: one spec row per request, null rows
    without a running slot, running slots a permutation of twice as many,
    num_computed drawn below 64, num_sampled the first step's accepted
    counts.  A few bytes per row: the launch is bound by its latency, not by
    HBM."""
    from linear_attention_speculative_kda_gb300 import api
    B = wl.spec.B
    gen = torch.Generator().manual_seed(19)
    idx = torch.randperm(2 * B, generator=gen)[:B].to(torch.int32)
    idx = torch.where(wl.state_indices > 0, idx, torch.full_like(idx, -1))
    num_computed = torch.randint(0, 64, (B,), generator=gen, dtype=torch.int32)
    num_sampled = wl.steps[0].num_accepted.clamp(min=0).to(torch.int32)
    i32 = dict(dtype=torch.int32, device=device)
    d_idx, d_ns, d_nc = idx.to(**i32), num_sampled.to(**i32), num_computed.to(**i32)
    col = torch.zeros(2 * B, **i32)
    acc = torch.zeros(2 * B, **i32)
    err = torch.zeros(1, **i32)

    def launch(_k):
        api.kda_record_state_blocks(d_idx, d_ns, d_nc, col, acc, block_size=16,
                                    block_table_width=8, error_word=err)

    us, how = time_launches(launch, iters, warmup)
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())} in record_state_blocks")
    b = record_blocks_bytes(idx.tolist())
    return {"rows": B, "timing": how, "launches": iters, "avg_us": us, "bytes_per_launch": b,
            "bound": "latency"}


def measure_commit_align(wl: W.Workload, device, iters: int, warmup: int, peak: float):
    """The align-mode commit on the workload's rows, timed alone: a pool with
    the row checkpoints and two blocks per request (block size 16; each
    request's num_computed drawn so that some steps cross a block boundary),
    records from one verify of the first step; timed from a CUDA graph
    replay."""
    from linear_attention_speculative_kda_gb300 import api
    sp = wl.spec
    B, H, D = sp.B, sp.H, sp.D
    width, bs = 2, 16
    S = 1 + B + B * width
    gen = torch.Generator().manual_seed(17)
    i32 = dict(dtype=torch.int32, device=device)
    pool = torch.empty((S, H, D, D), dtype=torch.float32, device=device).normal_(0.0, 0.05)
    slots = torch.where(wl.state_indices > 0, torch.arange(1, B + 1, dtype=torch.int32),
                        torch.zeros(B, dtype=torch.int32))
    table = (1 + B + torch.arange(B * width, dtype=torch.int32)).reshape(B, width)
    num_computed = torch.randint(0, bs, (B,), generator=gen, dtype=torch.int32)
    st = wl.steps[0]
    records = api.allocate_records(H, sp.Q, sp.record_slots, device)
    out = torch.empty((wl.total_tokens, H, D), dtype=torch.bfloat16, device=device)
    qkv, beta, g_raw = st.qkv.to(device), st.beta_buf.to(device), st.g_raw.to(device)
    cu, dslots = wl.cu_seqlens.to(**i32), slots.to(**i32)
    A_log, g_bias = wl.A_log.to(device), wl.g_bias.to(device)
    rr = None if wl.record_rows is None else wl.record_rows.to(**i32)
    kw = dict(window=sp.Q, record_slots=sp.record_slots,
              lower_bound=sp.lower_bound if sp.bounded else None)
    api.kda_verify(qkv[:, 0], qkv[:, 1], qkv[:, 2], g_raw, beta[:, :H], A_log, g_bias, pool, cu,
                   dslots, records, out, record_rows=rr, **kw)
    acc = st.num_accepted.to(**i32)
    dtable, dnc = table.to(**i32), num_computed.to(**i32)
    err = torch.zeros(1, **i32)

    def launch(_k):
        api.kda_commit_align(A_log, g_bias, pool, cu, dslots, acc, records, dtable, dnc,
                             block_size=bs, record_rows=rr, error_word=err, **kw)

    us, how = time_launches(launch, iters, warmup)
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())} in the align commit")
    b = align_commit_bytes(wl, table, num_computed.tolist(), bs, st.num_accepted.tolist())
    del pool, records
    return {"blocks_per_request": width, "block_size": bs, "timing": how, "launches": iters,
            "avg_us": us,
            "bytes_per_launch": b, "gbs": b / (us / 1e6) / 1e9,
            "frac": b / (us / 1e6) / 1e9 / peak}


def conv_align_bytes(wl: W.Workload, num_computed, block_size: int, acc, conv_dim: int,
                     hist: int, elem_bytes: int) -> int:
    """Algorithmic bytes of one align-mode conv compaction: every committing
    row reads its window at column n - 1 and writes it to its final block,
    and, when the step passes the next block boundary before its last token
    (a boundary block other than the final one), reads the window at column
    boundary_len - 1 and writes it to the boundary block."""
    lens = (wl.cu_seqlens[1:] - wl.cu_seqlens[:-1]).tolist()
    slots = wl.state_indices.tolist()
    windows = 0
    for b in range(wl.spec.B):
        n = min(max(int(acc[b]), 0), lens[b], wl.spec.Q)
        if slots[b] <= 0 or n <= 0:
            continue
        c = int(num_computed[b])
        windows += 2 if c + n > (c // block_size + 1) * block_size else 1
    return windows * 2 * conv_dim * hist * elem_bytes


def measure_conv_compact_align(wl: W.Workload, device, iters: int, warmup: int, peak: float):
    """The align-mode conv compaction on the workload's rows, timed alone:
    the bf16 channel-major conv pool with the rows' source slots and two
    blocks per request, block size 16 and num_computed drawn as in
    measure_commit_align; timed from a CUDA graph replay."""
    from linear_attention_speculative_kda_gb300 import api
    sp = wl.spec
    B = sp.B
    _, C, wconv = W.conv_shape(sp)
    width, bs = 2, 16
    S = 1 + B + B * width
    gen = torch.Generator().manual_seed(17)
    i32 = dict(dtype=torch.int32, device=device)
    pool = W.conv_state(S, C, wconv, seed=3).to(device)
    slots = torch.where(wl.state_indices > 0, torch.arange(1, B + 1, dtype=torch.int32),
                        torch.zeros(B, dtype=torch.int32))
    table = (1 + B + torch.arange(B * width, dtype=torch.int32)).reshape(B, width)
    num_computed = torch.randint(0, bs, (B,), generator=gen, dtype=torch.int32)
    cu, dslots = wl.cu_seqlens.to(**i32), slots.to(**i32)
    acc = wl.steps[0].num_accepted.to(**i32)
    dtable, dnc = table.to(**i32), num_computed.to(**i32)
    err = torch.zeros(1, **i32)

    def launch(_k):
        api.kda_conv_compact_align(pool, cu, dslots, acc, dtable, dnc, block_size=bs,
                                   window=sp.Q, error_word=err)

    us, how = time_launches(launch, iters, warmup)
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())} in the align conv compaction")
    b = conv_align_bytes(wl, num_computed.tolist(), bs, wl.steps[0].num_accepted.tolist(), C,
                         wconv - sp.Q + 1, 2)
    del pool
    return {"shape": [S, C, wconv], "dtype": "bf16", "layout": "channel-major",
            "blocks_per_request": width, "block_size": bs, "timing": how, "launches": iters,
            "avg_us": us, "bytes_per_launch": b, "gbs": b / (us / 1e6) / 1e9,
            "frac": b / (us / 1e6) / 1e9 / peak}


def run_ours(args):
    rank, world, local = dist_env()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    init_dist(world, "nccl")
    wl = W.generate(args.config, seed=shard_seed(args.seed, rank))
    eng = Engine(wl, device, args.records)
    names = [n for n, _ in eng.launches()]
    nl = len(names)
    bytes_per = dict(plan_bytes(wl, args.records))

    clocks = ClockSampler(local).__enter__()
    for _ in range(args.warmup):
        eng.run_step()
    torch.cuda.synchronize()
    if int(eng.err.item()) != 0:
        raise RuntimeError(f"device error word {int(eng.err.item())} during warm-up")

    stream = torch.cuda.current_stream(device)
    events = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(nl)] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_start = time.time()
    start.record(stream)
    for k in range(args.steps):
        eng.run_step()       # back to back, as a serving loop issues them
    stop.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms_total = start.elapsed_time(stop)
    ms_total = max_over_ranks(ms_total, world, device)
    # per-launch durations: the same K steps again with an event pair around
    # every launch (the pairs keep a launch from starting its set-up while
    # the previous one drains, so they are kept out of the pass above)
    for k in range(args.steps):
        eng.run_step(events[k])
    torch.cuda.synchronize()
    clocks.mark(t_start, time.time())
    clocks.__exit__(None, None, None)
    per_kernel = {n: [] for n in names}
    for k in range(args.steps):
        for i, n in enumerate(names):
            per_kernel[n].append(events[k][i][0].elapsed_time(events[k][i][1]))
    if int(eng.err.item()) != 0:
        raise RuntimeError(f"device error word {int(eng.err.item())}")

    units = units_per_step(wl) * args.steps
    units_all = sum_over_ranks(units, world, device)
    value = units_all / (ms_total / 1e3)
    ms_per_step = ms_total / args.steps

    peak, peak_src = hbm_peak()
    clock_summary = clocks.summary()
    ops_per = dict(plan_fp32_ops(wl, args.records))
    kernels = []
    for n in names:
        avg_ms = statistics.mean(per_kernel[n])
        b = bytes_per[n]
        kernels.append({"name": n, "launches": args.steps, "avg_us": avg_ms * 1e3,
                        "median_us": statistics.median(per_kernel[n]) * 1e3,
                        "bytes_per_launch": b, "gbs": b / (avg_ms / 1e3) / 1e9,
                        "fp32_ops_per_launch": ops_per[n],
                        "share": sum(per_kernel[n]) / max(1e-9, sum(sum(v) for v in
                                                                  per_kernel.values()))})
    dom = max(kernels, key=lambda x: x["share"])
    traffic, traffic_src = profiled_traffic(
        dom["name"], wl.spec.name if args.records == "raw" else f"{wl.spec.name}_{args.records}")
    step_bytes = sum(bytes_per.values())
    roofline = {"bound": "hbm", "kernel": dom["name"], "achieved": dom["gbs"], "peak": peak,
                "unit": "GB/s", "frac": dom["gbs"] / peak,
                "peak_source": f"{peak_src} ({'of measured' if peak_src == 'measured' else 'of fallback'})",
                "traffic": traffic, "traffic_source": traffic_src,
                "algorithmic_bytes_per_launch": dom["bytes_per_launch"]}
    # the FP32 pipe beside it, and the launch against the lower of the two roofs
    alu_peak, alu_src = fp32_peak(device, clock_summary)
    dom_s = dom["avg_us"] / 1e6
    t_hbm = dom["bytes_per_launch"] / (peak * 1e9)
    t_alu = dom["fp32_ops_per_launch"] / (alu_peak * 1e12)
    roofline["alu"] = {"ops_per_launch": dom["fp32_ops_per_launch"], "unit": "T ops/s",
                       "achieved": dom["fp32_ops_per_launch"] / dom_s / 1e12,
                       "peak": alu_peak, "frac": t_alu / dom_s, "peak_source": alu_src}
    roofline["min_roof"] = {"bound": "hbm" if t_hbm >= t_alu else "alu",
                            "roof_us": max(t_hbm, t_alu) * 1e6,
                            "frac": max(t_hbm, t_alu) / dom_s}
    step_gbs = step_bytes * args.steps / (ms_total / 1e3) / 1e9

    # end to end through the public API with host buffers: issued call by
    # call from the host, and the same steps replayed from a CUDA graph
    hio = HostIO(eng)
    hio.run(4)
    torch.cuda.synchronize()
    e_start, e_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    e_start.record(stream)
    hio.run(args.steps)
    e_stop.record(stream)
    torch.cuda.synchronize()
    e_ms = max_over_ranks(e_start.elapsed_time(e_stop), world, device)
    graph = hio.capture()
    g_steps = hio.graph_steps()
    replays = max(1, -(-args.steps // g_steps))
    hio.fill_first()
    graph.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e_start.record(stream)
    hio.fill_first()  # the first step's inputs, inside the timed region
    for _ in range(replays):
        graph.replay()
    e_stop.record(stream)
    torch.cuda.synchronize()
    g_ms = max_over_ranks(e_start.elapsed_time(e_stop), world, device) / (replays * g_steps)
    del graph
    units_step = units_all / args.steps
    # both ways of issuing the same steps through the public API; the line's
    # figure is the faster one, named in `issue`
    ways = [{"value": units_all / (e_ms / 1e3), "ms_per_step": e_ms / args.steps,
             "issue": "call by call from the host"},
            {"value": units_step / (g_ms / 1e3), "ms_per_step": g_ms,
             "issue": f"CUDA graph of {g_steps} pipelined steps, replayed {replays} times"}]
    best = min(ways, key=lambda w: w["ms_per_step"])
    e2e = {"value": best["value"], "unit": UNIT, "h2d_bytes_per_step": hio.h2d,
           "d2h_bytes_per_step": hio.d2h, "ms_per_step": best["ms_per_step"],
           "issue": best["issue"], "host_issued": ways[0], "graph": ways[1]}

    # the commit's conv-state compaction, a separate launch, timed on its own
    conv = None
    if not args.no_extras:
        conv = {lay: measure_conv_compact(wl, device, max(20, args.steps // 4), args.warmup,
                                          peak, layout=lay) for lay in ("dim_first", "col_first")}

    # the align-mode (paged-block) commit on the same rows, timed on its own
    del hio
    align = record = flush = conv_align = None
    if not args.no_extras:
        align = measure_commit_align(wl, device, max(20, args.steps // 4), args.warmup, peak)
        conv_align = measure_conv_compact_align(wl, device, max(20, args.steps // 4),
                                                args.warmup, peak)
        record = measure_record_state_blocks(wl, device, max(20, args.steps // 4), args.warmup)
        if wl.spec.deferred:
            flush = measure_flush(wl, device, max(20, args.steps // 4), args.warmup, peak,
                                  args.records)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, args.cpu_budget, args.records)

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded)", "config": workload_config(wl, world, args.records),
            "hbm_gbs_step": step_gbs, "hbm_frac_step": step_gbs / peak,
            "roofline": roofline, "kernels": kernels,
            "kernel_timing": "per-launch CUDA events over a second pass of the same steps",
            "gpu_launches": nl * args.steps,
            "e2e": e2e, "clocks": clock_summary, "cpu_baseline": cpu,
            "extras": None if args.no_extras else {"conv_compact": conv,
                                                   "commit_align": align,
                                                   "conv_compact_align": conv_align,
                                                   "record_state_blocks": record,
                                                   "flush": flush}}
    if world > 1:
        torch.distributed.barrier()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    wl = W.generate(args.config, seed=args.seed)
    threads = max(1, os.cpu_count() or 1)
    rng = np.random.default_rng(7)
    rows_per_step = max(1, min(wl.spec.B, args.reference_rows))
    times, units = [], 0
    for k in range(args.warmup + args.steps):
        rows = sorted(rng.choice(wl.spec.B, size=rows_per_step, replace=False).tolist())
        u, dt = oracle_sample_run(wl, rows, threads, args.records)
        if k >= args.warmup:
            times.append(dt)
            units += u
    secs = sum(times)
    value = units / secs
    sample = (f"{rows_per_step} of {wl.spec.B} rows x {wl.spec.H} heads x {wl.spec.steps} "
              f"decode step(s) per step, fp64 C oracle, {threads} threads")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded)",
            "config": workload_config(wl, 1, args.records),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="deferred2", choices=sorted(W.CONFIGS))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the separately timed conv compactions, align commit, "
                         "running state column and flush")
    ap.add_argument("--reference-rows", type=int, default=8)
    ap.add_argument("--records", choices=["raw", "correction"], default="raw",
                    help="record format: raw inputs replayed (default) or fp32 deltas folded")
    ap.add_argument("--ncu-traffic", metavar="CSV",
                    help="write profiles/ncu_<config>.json from an ncu --csv log of one "
                         "step's launches (dram__bytes_read.sum, dram__bytes_write.sum, "
                         "--print-units base) and exit")
    ap.add_argument("--ncu-command", default="",
                    help="the ncu command line that made --ncu-traffic's log")
    args = ap.parse_args(argv)
    if args.ncu_traffic:
        wl = W.generate(args.config, seed=args.seed, pool=False)
        name = args.config if args.records == "raw" else f"{args.config}_{args.records}"
        print(write_traffic(args.ncu_traffic, name, launch_names(wl), args.ncu_command))
        return
    args.warmup = max(3, args.warmup)   # at least 3 untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
