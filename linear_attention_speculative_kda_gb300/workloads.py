"""Seeded synthetic workloads for KDA speculative verify/commit.

This module only draws random inputs and lays them out; it holds none of the
method's arithmetic and imports neither the CUDA binding nor the oracle, so
that both sides can be fed the same bytes.

Shapes and distributions follow the workloads the pages run: head dim 128,
fp32 recurrent state, bf16 activations, a window of 1 + num_spec tokens with
num_spec in 1..7 (the PR's eligibility list: MTP/DFlash depth 1-7).  Every
tensor is drawn from one CPU ``torch.Generator`` in a fixed order, values in
fp32 and cast to bf16 with round-to-nearest-even.

Activation layout mirrors the layer (kda.py, ``forward``/``_forward``): q, k
and v are strided views into one merged ``[T, 3, H, D]`` buffer (token
stride 3*H*D), beta_raw is a strided view into a ``[T, H + 8]`` buffer, and
g_raw is contiguous ``[T, H, D]``.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import torch

HEAD_DIM = 128


@dataclass(frozen=True)
class Spec:
    """A workload: batch shape, pool sizes and the structure of the rows."""

    name: str
    B: int                    # request rows
    H: int                    # heads
    Q: int                    # record window, 1 + num_spec
    S: int                    # state-pool slots (slot 0 is the null block)
    R: int = 0                # record slots (0: one per row, R = B)
    lens: str = "fixed"       # "fixed": every row has Q tokens; "uniform": U{1..Q}
    bounded: bool = False     # bounded sigmoid gate
    lower_bound: float = -5.0
    null_rows: int = 0        # rows whose state index is 0 (skipped)
    deferred: bool = False    # record_rows permutation + eager mask
    eager_prob: float = 0.1
    steps: int = 1
    slot_mode: str = "distinct"  # "distinct": B slots from 1..S-1; "perm": 1..B
    D: int = HEAD_DIM

    @property
    def record_slots(self) -> int:
        return self.R if self.R else self.B


# The five workloads the benchmark and the parity tests use.
CONFIGS: dict[str, Spec] = {
    # B=4, H=4, Q=4 (1+3 drafts), 8-slot pool, accepted U{0..4}.
    "tiny": Spec("tiny", B=4, H=4, Q=4, S=8, slot_mode="perm"),
    # MTP3 decode: B=64, H=32, Q=4, slots a permutation of 1..64 in a
    # 96-slot pool.
    "mtp3": Spec("mtp3", B=64, H=32, Q=4, S=96, slot_mode="perm"),
    # DFlash depth 7 with the bounded gate (lower bound -5); 10% of rows
    # (26 of 256) carry the null state index.
    "dflash7": Spec("dflash7", B=256, H=16, Q=8, S=320, bounded=True,
                    lower_bound=-5.0, null_rows=26),
    # Mixed varlen: B=512, H=32, per-row length U{1..8}, 768-slot pool.
    "mixed": Spec("mixed", B=512, H=32, Q=8, S=768, lens="uniform"),
    # Deferred commit over two chained steps: B=1024, H=16, Q=4, record
    # rows a permutation of 0..1023, 10% of rows committed eagerly.
    "deferred2": Spec("deferred2", B=1024, H=16, Q=4, S=1280, R=1024,
                      deferred=True, eager_prob=0.1, steps=2),
}


@dataclass
class StepInputs:
    """One step's activations and accepted counts (CPU tensors)."""

    qkv: torch.Tensor        # [T, 3, H, D] bf16, owns q, k, v
    beta_buf: torch.Tensor   # [T, H + 8] bf16, owns beta_raw
    g_raw: torch.Tensor      # [T, H, D] bf16 contiguous
    num_accepted: torch.Tensor  # [B] int32
    eager: torch.Tensor | None  # [B] uint8 or None

    @property
    def q(self):
        return self.qkv[:, 0]

    @property
    def k(self):
        return self.qkv[:, 1]

    @property
    def v(self):
        return self.qkv[:, 2]

    @property
    def beta_raw(self):
        return self.beta_buf[:, : self.qkv.shape[2]]


@dataclass
class Workload:
    spec: Spec
    A_log: torch.Tensor          # [H] fp32
    g_bias: torch.Tensor         # [H * D] fp32
    pool: torch.Tensor           # [S, H, D, D] fp32
    cu_seqlens: torch.Tensor     # [B + 1] int32
    state_indices: torch.Tensor  # [B] int32
    record_rows: torch.Tensor | None  # [B] int32 or None
    steps: list = field(default_factory=list)

    @property
    def lens(self) -> torch.Tensor:
        return self.cu_seqlens[1:] - self.cu_seqlens[:-1]

    @property
    def total_tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def scale(self) -> float:
        return self.spec.D ** -0.5


def _bf16_normal(shape, gen):
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def _step_inputs(spec: Spec, lens: torch.Tensor, gen) -> StepInputs:
    T = int(lens.sum())
    H, D = spec.H, spec.D
    qkv = _bf16_normal((T, 3, H, D), gen)
    beta_buf = _bf16_normal((T, H + 8), gen)
    g_raw = _bf16_normal((T, H, D), gen)
    # accepted counts U{0..len} per row
    hi = lens.to(torch.float64) + 1.0
    u = torch.rand(spec.B, generator=gen, dtype=torch.float64)
    num_accepted = torch.floor(u * hi).to(torch.int32)
    num_accepted = torch.minimum(num_accepted, lens.to(torch.int32))
    eager = None
    if spec.deferred:
        eager = (torch.rand(spec.B, generator=gen) < spec.eager_prob).to(torch.uint8)
    return StepInputs(qkv, beta_buf, g_raw, num_accepted, eager)


def generate(spec: Spec | str, seed: int = 0, *, pool: bool = True) -> Workload:
    """Draw a workload.  ``pool=False`` leaves the state pool empty (zeros of
    the right shape are NOT allocated; ``Workload.pool`` is then None)."""
    if isinstance(spec, str):
        spec = CONFIGS[spec]
    gen = torch.Generator().manual_seed(seed)
    B, H, D, Q, S = spec.B, spec.H, spec.D, spec.Q, spec.S
    if B + 1 > S and B > 0:
        raise ValueError("pool too small for distinct slots")

    # Row lengths and varlen offsets.
    if spec.lens == "fixed":
        lens = torch.full((B,), Q, dtype=torch.int64)
    elif spec.lens == "uniform":
        lens = torch.randint(1, Q + 1, (B,), generator=gen, dtype=torch.int64)
    else:
        raise ValueError(spec.lens)
    cu = torch.zeros(B + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(lens, 0)

    # Distinct state slots drawn from 1..S-1, then the null rows.
    if spec.slot_mode == "perm":
        slots = torch.randperm(B, generator=gen) + 1
    else:
        slots = torch.randperm(S - 1, generator=gen)[:B] + 1
    if spec.null_rows:
        null = torch.randperm(B, generator=gen)[: spec.null_rows]
        slots[null] = 0

    record_rows = None
    if spec.deferred:
        record_rows = torch.randperm(spec.record_slots, generator=gen)[:B].to(torch.int32)

    A_log = torch.rand(H, generator=gen, dtype=torch.float32) * 2.7
    g_bias = torch.randn(H * D, generator=gen, dtype=torch.float32) * 0.1
    pool_t = None
    if pool:
        pool_t = torch.randn((S, H, D, D), generator=gen, dtype=torch.float32) * 0.05

    wl = Workload(spec=spec, A_log=A_log, g_bias=g_bias, pool=pool_t,
                  cu_seqlens=cu.to(torch.int32), state_indices=slots.to(torch.int32),
                  record_rows=record_rows)
    for _ in range(spec.steps):
        wl.steps.append(_step_inputs(spec, lens, gen))
    return wl


def custom(B: int, H: int, Q: int, lens, *, S: int | None = None, R: int = 0,
           slots=None, bounded: bool = False, lower_bound: float = -5.0,
           deferred: bool = False, eager_prob: float = 0.1, steps: int = 1,
           seed: int = 0, record_rows=None, pool_std: float = 0.05) -> Workload:
    """A small workload with explicit row lengths and slots (edge cases:
    empty rows, ragged lengths, null rows, out-of-range metadata)."""
    lens = torch.as_tensor(lens, dtype=torch.int64)
    assert lens.numel() == B
    if S is None:
        S = B + 2
    spec = Spec("custom", B=B, H=H, Q=Q, S=S, R=R, bounded=bounded,
                lower_bound=lower_bound, deferred=deferred,
                eager_prob=eager_prob, steps=steps)
    gen = torch.Generator().manual_seed(seed)
    D = spec.D
    cu = torch.zeros(B + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(lens.clamp(min=0), 0)
    if slots is None:
        slots = torch.randperm(S - 1, generator=gen)[:B] + 1
    slots = torch.as_tensor(slots, dtype=torch.int32)
    if record_rows is None and deferred:
        record_rows = torch.randperm(spec.record_slots, generator=gen)[:B]
    if record_rows is not None:
        record_rows = torch.as_tensor(record_rows, dtype=torch.int32)
    A_log = torch.rand(H, generator=gen, dtype=torch.float32) * 2.7
    g_bias = torch.randn(H * D, generator=gen, dtype=torch.float32) * 0.1
    pool_t = torch.randn((S, H, D, D), generator=gen, dtype=torch.float32) * pool_std
    wl = Workload(spec=spec, A_log=A_log, g_bias=g_bias, pool=pool_t,
                  cu_seqlens=cu.to(torch.int32), state_indices=slots,
                  record_rows=record_rows)
    lens_pos = lens.clamp(min=0)
    for _ in range(steps):
        wl.steps.append(_step_inputs(spec, lens_pos, gen))
    return wl


# ------------------------------------------------------------ conv state --

CONV_KERNEL = 4   # short causal conv width (history 3), the usual KDA setting


def conv_shape(spec: Spec, kernel: int = CONV_KERNEL) -> tuple[int, int, int]:
    """[S, conv_dim, width] of the conv-state pool of a workload: one conv
    channel per q, k and v channel of every head (conv_dim = 3 * H * D) and
    kernel - 1 history columns plus Q - 1 draft columns."""
    return spec.S, 3 * spec.H * spec.D, kernel - 1 + spec.Q - 1


def conv_state(S: int, conv_dim: int, width: int, *, dtype=torch.bfloat16, seed: int = 0,
               layout: str = "dim_first") -> torch.Tensor:
    """A seeded conv-state pool viewed as [S, conv_dim, width] (CPU).
    ``dim_first``: stored channel-major, [S][conv_dim][width];
    ``col_first``: stored column-major, [S][width][conv_dim], viewed
    transposed.  Values are N(0, 1) cast to ``dtype`` (only their bits
    matter: the compaction moves them)."""
    gen = torch.Generator().manual_seed(seed)
    if layout == "dim_first":
        return torch.randn((S, conv_dim, width), generator=gen).to(dtype)
    if layout == "col_first":
        return torch.randn((S, width, conv_dim), generator=gen).to(dtype).transpose(1, 2)
    raise ValueError(layout)
