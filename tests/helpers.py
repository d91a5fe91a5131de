"""Test helpers: feed one seeded workload to both the oracle and the library.

The conversions here are exact (bf16 and fp32 values widened to float64);
no arithmetic of the method happens in this file.
"""

from __future__ import annotations

import numpy as np
import torch

from linear_attention_speculative_kda_gb300 import workloads as W
from oracle import kda_oracle as O


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


def oracle_layer(wl: W.Workload) -> O.Layer:
    sp = wl.spec
    return O.Layer(num_heads=sp.H, head_dim=sp.D, window=sp.Q, a_log=f64(wl.A_log),
                   g_bias=f64(wl.g_bias).reshape(sp.H, sp.D), bounded=sp.bounded,
                   lower_bound=sp.lower_bound if sp.bounded else 0.0, scale=wl.scale)


def oracle_step(wl: W.Workload, step: int = 0, cu_seqlens=None, state_indices=None,
                record_rows="default") -> O.Step:
    st = wl.steps[step]
    rr = wl.record_rows if isinstance(record_rows, str) else record_rows
    return O.Step(q=f64(st.q), k=f64(st.k), v=f64(st.v), g_raw=f64(st.g_raw),
                  beta_raw=f64(st.beta_raw),
                  cu_seqlens=(wl.cu_seqlens if cu_seqlens is None else cu_seqlens).numpy(),
                  state_indices=(wl.state_indices if state_indices is None
                                 else state_indices).numpy(),
                  record_rows=None if rr is None else np.asarray(rr))


def oracle_cache(wl: W.Workload, record_format: str = "raw") -> O.Cache:
    return O.Cache(wl.pool.numpy(), wl.spec.record_slots, record_format=record_format)


# --------------------------------------------------------------- GPU side --

class DeviceRun:
    """Device copies of a workload plus the buffers the library writes."""

    def __init__(self, wl: W.Workload, device="cuda", with_traj=False, sentinel=True,
                 record_format="raw"):
        from linear_attention_speculative_kda_gb300 import api
        sp = wl.spec
        self.wl = wl
        self.record_format = record_format
        self.dev = torch.device(device)
        d = self.dev
        self.A_log = wl.A_log.to(d)
        self.g_bias = wl.g_bias.to(d)
        self.pool = wl.pool.to(d)
        self.pool0 = self.pool.clone()
        self.cu = wl.cu_seqlens.to(d)
        self.slots = wl.state_indices.to(d)
        self.record_rows = None if wl.record_rows is None else wl.record_rows.to(d)
        self.steps = []
        for st in wl.steps:
            self.steps.append(dict(
                qkv=st.qkv.to(d), beta_buf=st.beta_buf.to(d), g_raw=st.g_raw.to(d),
                num_accepted=st.num_accepted.to(d),
                eager=None if st.eager is None else st.eager.to(d)))
        T = wl.total_tokens
        self.records = api.allocate_records(sp.H, sp.Q, sp.record_slots, d,
                                            record_format=record_format)
        self.out = torch.empty((T, sp.H, sp.D), dtype=torch.bfloat16, device=d)
        if sentinel:
            self.records.fill_(-7.0)
            self.out.fill_(-9.0)
        self.traj = (torch.full((T, sp.H, sp.D, sp.D), float("nan"), device=d)
                     if with_traj else None)
        self.pending = torch.zeros(sp.record_slots, dtype=torch.int32, device=d)
        self.err = torch.zeros(1, dtype=torch.int32, device=d)

    def kw(self):
        sp = self.wl.spec
        return dict(window=sp.Q, record_slots=sp.record_slots,
                    lower_bound=sp.lower_bound if sp.bounded else None,
                    record_format=self.record_format)

    def verify(self, step=0, pending=False, cu=None, slots=None, record_rows="default"):
        from linear_attention_speculative_kda_gb300 import api
        s = self.steps[step]
        H = self.wl.spec.H
        rr = self.record_rows if isinstance(record_rows, str) else record_rows
        api.kda_verify(s["qkv"][:, 0], s["qkv"][:, 1], s["qkv"][:, 2], s["g_raw"],
                       s["beta_buf"][:, :H], self.A_log, self.g_bias, self.pool,
                       self.cu if cu is None else cu, self.slots if slots is None else slots,
                       self.records, self.out, record_rows=rr,
                       pending=self.pending if pending else None, trajectory_out=self.traj,
                       error_word=self.err, **self.kw())
        return self.out

    def commit(self, step=0, deferred=False, eager="default", num_accepted=None, cu=None,
               slots=None, record_rows="default"):
        from linear_attention_speculative_kda_gb300 import api
        s = self.steps[step]
        rr = self.record_rows if isinstance(record_rows, str) else record_rows
        em = s["eager"] if isinstance(eager, str) else eager
        api.kda_commit(self.A_log, self.g_bias, self.pool, self.cu if cu is None else cu,
                       self.slots if slots is None else slots,
                       s["num_accepted"] if num_accepted is None else num_accepted,
                       self.records, record_rows=rr, pending=self.pending if deferred else None,
                       eager=em if deferred else None, error_word=self.err, **self.kw())

    def flush(self, slots=None, record_rows="default"):
        from linear_attention_speculative_kda_gb300 import api
        rr = self.record_rows if isinstance(record_rows, str) else record_rows
        api.kda_flush(self.A_log, self.g_bias, self.pool, self.slots if slots is None else slots,
                      self.records, self.pending, record_rows=rr, error_word=self.err,
                      **self.kw())


# bf16 outputs.  The stated tolerance is an absolute 2e-3 element by element.
# At these workloads' output scale (median |o| about 1e-3) that bound alone
# would pass a wrong output, so the check also holds every element to what
# rounding allows: the kernel rounds an fp32 value to bf16 (at most half a
# bf16 ulp) and its fp32 arithmetic differs from the double-precision oracle
# by far less than OUT_FLOOR (about 6e-10 at most on the five workloads).
OUT_ATOL = 2e-3
OUT_ULPS = 0.5
OUT_FLOOR = 1e-7


def bf16_ulp(x) -> np.ndarray:
    """Spacing of bfloat16 numbers at |x| (8 significant bits):
    2^(floor(log2 |x|) - 7); 2^-133 (the smallest subnormal step) at 0."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(ax)                       # ax = m * 2^e with m in [0.5, 1)
    return np.where(ax > 0, np.ldexp(1.0, e - 8), np.ldexp(1.0, -133))


def out_errors(got, oracle_out: np.ndarray):
    """(|got - oracle|, |got - oracle| in bf16 ulps of the oracle value) on
    the entries the oracle wrote (NaN elsewhere)."""
    g = f64(got) if isinstance(got, torch.Tensor) else np.asarray(got, dtype=np.float64)
    mask = ~np.isnan(oracle_out)
    assert mask.any()
    diff = np.abs(g[mask] - oracle_out[mask])
    return diff, diff / bf16_ulp(oracle_out[mask]), oracle_out[mask]


def assert_out_close(gpu_out, oracle_out: np.ndarray, rows_tokens=None, atol=OUT_ATOL,
                     ulps=OUT_ULPS, floor=OUT_FLOOR):
    """bf16 outputs against the unrounded double-precision oracle, element by
    element: |gpu - oracle| <= 2e-3 (the stated tolerance) and
    |gpu - oracle| <= 0.5 bf16 ulp of |oracle| + 1e-7 (the rounding bound).
    Returns the worst error in bf16 ulps."""
    diff, in_ulps, ref = out_errors(gpu_out, oracle_out)
    assert diff.max() <= atol, f"max |out - oracle| = {diff.max():.3e} > {atol}"
    bound = ulps * bf16_ulp(ref) + floor
    bad = diff > bound
    if bad.any():
        i = int(np.argmax(diff - bound))
        raise AssertionError(
            f"{int(bad.sum())} of {diff.size} outputs differ from the oracle by more than "
            f"{ulps} bf16 ulp + {floor:g}; worst: |d| = {diff[i]:.3e} at oracle value "
            f"{ref[i]:.6e} ({in_ulps[i]:.2f} ulp)")
    return float(in_ulps.max())


def assert_state_close(gpu_tile: np.ndarray, oracle_tile: np.ndarray, rel=1e-5):
    """fp32 states, normwise per (slot, head) tile:
    max |gpu - oracle| <= rel * max |oracle|."""
    err = np.abs(gpu_tile - oracle_tile).max()
    ref = np.abs(oracle_tile).max()
    assert err <= rel * ref, f"state error {err:.3e} > {rel} * {ref:.3e}"
    return float(err / ref) if ref > 0 else 0.0
