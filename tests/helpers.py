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


def oracle_cache(wl: W.Workload) -> O.Cache:
    return O.Cache(wl.pool.numpy(), wl.spec.record_slots)
