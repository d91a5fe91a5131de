"""Thin ctypes binding of ``libkda.so`` (the C ABI of ``include/kda.h``).

Argument marshalling only: every function checks dtypes, devices and shapes
of the torch tensors it is given, fills a ``kda_config`` and passes raw
device pointers and the current CUDA stream to the entry point of the same
name.  Every step of the method runs in the library's CUDA kernels; there is
no fallback of any kind.  If the library has not been built, the first call
raises.
"""

from __future__ import annotations

import ctypes
import functools
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIBRARY = os.path.join(_PKG, "libkda.so")

HEAD_DIM = 128
MAX_WINDOW = 8
RECORD_STRIDE = 392          # bf16 elements per token record (k, v, g, beta, pad)
CORRECTION_RECORD_BYTES = 1024  # fp32 delta, bf16 k, bf16 g_raw per token
RECORD_FORMATS = {"raw": 0, "correction": 1}

KDA_OK = 0
KDA_ERR_INVALID_ARG = 1
KDA_ERR_UNSUPPORTED = 2
KDA_ERR_CUDA = 3

ROW_BAD_LENGTH = 1
ROW_BAD_SLOT = 2
ROW_BAD_RECORD = 4
ROW_BAD_PENDING = 8
ERR_WAIT_TIMEOUT = 16
ROW_BAD_BLOCK = 32

EXPORTED = (
    "kda_records_bytes",
    "kda_correction_records_bytes",
    "kda_verify",
    "kda_commit",
    "kda_flush",
    "kda_conv_compact",
    "kda_commit_align",
    "kda_conv_compact_align",
    "kda_record_state_blocks",
    "kda_status_string",
    "kda_abi_version",
)


class KDAError(RuntimeError):
    """A call into libkda returned a status other than KDA_OK."""

    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: status {status} ({_status_name(status)})")
        self.status = status


class KdaConfig(ctypes.Structure):
    _fields_ = [
        ("num_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("window", ctypes.c_int32),
        ("num_slots", ctypes.c_int32),
        ("record_slots", ctypes.c_int32),
        ("use_lower_bound", ctypes.c_int32),
        ("lower_bound", ctypes.c_float),
        ("scale", ctypes.c_float),
        ("stride_q_t", ctypes.c_int64),
        ("stride_k_t", ctypes.c_int64),
        ("stride_v_t", ctypes.c_int64),
        ("stride_g_t", ctypes.c_int64),
        ("stride_beta_t", ctypes.c_int64),
        ("record_format", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]


class KdaConvConfig(ctypes.Structure):
    _fields_ = [
        ("num_slots", ctypes.c_int32),
        ("conv_dim", ctypes.c_int32),
        ("width", ctypes.c_int32),
        ("window", ctypes.c_int32),
        ("elem_bytes", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
        ("stride_slot", ctypes.c_int64),
        ("stride_dim", ctypes.c_int64),
        ("stride_col", ctypes.c_int64),
    ]


MAX_CONV_HISTORY = 16


class KdaAlign(ctypes.Structure):
    _fields_ = [
        ("block_table", ctypes.c_void_p),
        ("block_table_stride", ctypes.c_int64),
        ("block_table_width", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("num_requests", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
        ("num_computed", ctypes.c_void_p),
        ("request_indices", ctypes.c_void_p),
    ]

_lib_handle = None


def library_path() -> str:
    return _LIBRARY


def load_library():
    """Load libkda.so (once).  Raises if it is missing: there is no fallback."""
    global _lib_handle
    if _lib_handle is not None:
        return _lib_handle
    if not os.path.exists(_LIBRARY):
        raise RuntimeError(
            f"libkda.so not found at {_LIBRARY}; build it first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    _lib_handle = bind_library(_LIBRARY)
    return _lib_handle


def bind_library(path: str):
    """A ctypes handle of a build of the library at ``path`` (libkda.so, or a
    test variant from build.build_variant) with every entry point's argument
    types declared."""
    lib = ctypes.CDLL(path)
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    cfgp = ctypes.POINTER(KdaConfig)
    lib.kda_records_bytes.restype = ctypes.c_size_t
    lib.kda_records_bytes.argtypes = [i32, i32, i32]
    lib.kda_correction_records_bytes.restype = ctypes.c_size_t
    lib.kda_correction_records_bytes.argtypes = [i32, i32, i32]
    lib.kda_verify.restype = ctypes.c_int
    lib.kda_verify.argtypes = [cfgp] + [vp] * 10 + [i32] + [vp] * 7
    lib.kda_commit.restype = ctypes.c_int
    lib.kda_commit.argtypes = [cfgp] + [vp] * 5 + [i32] + [vp] * 7
    lib.kda_flush.restype = ctypes.c_int
    lib.kda_flush.argtypes = [cfgp] + [vp] * 4 + [i32] + [vp] * 5
    lib.kda_conv_compact.restype = ctypes.c_int
    lib.kda_conv_compact.argtypes = [ctypes.POINTER(KdaConvConfig)] + [vp] * 3 + [i32] + [vp] * 3
    alp = ctypes.POINTER(KdaAlign)
    lib.kda_commit_align.restype = ctypes.c_int
    lib.kda_commit_align.argtypes = [cfgp] + [vp] * 5 + [i32] + [vp] * 3 + [alp, vp, vp, vp, vp]
    lib.kda_conv_compact_align.restype = ctypes.c_int
    lib.kda_conv_compact_align.argtypes = ([ctypes.POINTER(KdaConvConfig)] + [vp] * 3 + [i32] +
                                           [vp, alp, vp, vp])
    lib.kda_record_state_blocks.restype = ctypes.c_int
    lib.kda_record_state_blocks.argtypes = [alp, vp, vp, i32, vp, vp, i32, vp, vp]
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_status_string.argtypes = [ctypes.c_int]
    lib.kda_abi_version.restype = i32
    lib.kda_abi_version.argtypes = []
    return lib


def _status_name(status: int) -> str:
    try:
        return load_library().kda_status_string(status).decode()
    except Exception:  # pragma: no cover - only for messages
        return "?"


def _check(fn: str, status: int) -> None:
    if status != KDA_OK:
        raise KDAError(fn, status)


def _ptr(t):
    # a plain int: ctypes converts it for c_void_p parameters (None is NULL)
    return None if t is None else t.data_ptr()


def _stream_ptr(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _token_stride(t: torch.Tensor) -> int:
    # [T, H, D] (or [1, T, H, D]) activation with heads and channels packed
    if t.dim() == 4:
        t = t[0]
    if t.dim() == 3:
        if t.stride(2) != 1 or t.stride(1) != t.shape[2]:
            raise ValueError("activations need contiguous [H, D] inside a token")
    elif t.dim() == 2:
        if t.stride(1) != 1:
            raise ValueError("beta needs contiguous heads inside a token")
    else:
        raise ValueError("unexpected activation rank")
    return t.stride(0) if t.shape[0] > 1 else max(t.stride(0), 1)


def _req(t, dtype, name, device):
    if t is None:
        raise ValueError(f"{name} is required")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}")
    return t


def _opt(t, dtype, name, device):
    return None if t is None else _req(t, dtype, name, device)


# Shape and size checks.  The C ABI takes bare pointers and cannot see how
# large a buffer is, so the binding checks every tensor the kernels index
# against the sizes the call implies, before anything is launched.

def _tokens(t, name, H, D):
    """Token count of a [T, H, D] (or [1, T, H, D]) activation, or of a
    [T, H] (or [1, T, H]) one when D is None."""
    lead = 4 if D is not None else 3
    if t.dim() == lead:
        if t.shape[0] != 1:
            raise ValueError(f"{name}: a leading batch dimension must be 1")
        t = t[0]
    want = (H, D) if D is not None else (H,)
    if t.dim() != len(want) + 1 or tuple(t.shape[1:]) != want:
        shape = "[T, H, D]" if D is not None else "[T, H]"
        raise ValueError(f"{name} must be {shape} with H={H}" +
                         (f", D={D}" if D is not None else "") + f", got {tuple(t.shape)}")
    return t.shape[0]


def _at_least(t, n, name):
    if t is not None and t.numel() < n:
        raise ValueError(f"{name} needs at least {n} elements, has {t.numel()}")


def _check_pool(state_pool):
    if (state_pool.dim() != 4 or not state_pool.is_contiguous()
            or state_pool.shape[2] != state_pool.shape[3]):
        raise ValueError("state_pool must be a contiguous [S, H, V, K] tensor with V == K")
    return state_pool.shape[0], state_pool.shape[1], state_pool.shape[3]


def _check_gate(A_log, g_bias, H, D):
    if not A_log.is_contiguous() or not g_bias.is_contiguous():
        raise ValueError("A_log and g_bias must be contiguous")
    _at_least(A_log, H, "A_log")
    _at_least(g_bias, H * D, "g_bias")


def _check_rows(B, record_slots, record_rows=None, pending=None, eager=None, error_word=None):
    for name, t in (("record_rows", record_rows), ("pending", pending), ("eager", eager),
                    ("error_word", error_word)):
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    _at_least(record_rows, B, "record_rows")
    _at_least(pending, record_slots, "pending")
    _at_least(eager, B, "eager")
    _at_least(error_word, 1, "error_word")


def _format_code(record_format: str) -> int:
    try:
        return RECORD_FORMATS[record_format]
    except KeyError:
        raise ValueError(f"record_format must be one of {sorted(RECORD_FORMATS)}") from None


def make_config(num_heads, window, num_slots, record_slots, *, lower_bound=None,
                scale=None, strides=(1, 1, 1, 1, 1), head_dim=HEAD_DIM,
                record_format: str = "raw") -> KdaConfig:
    """A new ``kda_config`` (the entry points below share read-only cached
    ones, see ``_config``)."""
    cfg = KdaConfig()
    cfg.record_format = _format_code(record_format)
    cfg.reserved = 0
    cfg.num_heads = num_heads
    cfg.head_dim = head_dim
    cfg.window = window
    cfg.num_slots = num_slots
    cfg.record_slots = record_slots
    cfg.use_lower_bound = 0 if lower_bound is None else 1
    cfg.lower_bound = 0.0 if lower_bound is None else float(lower_bound)
    cfg.scale = head_dim ** -0.5 if scale is None else float(scale)
    (cfg.stride_q_t, cfg.stride_k_t, cfg.stride_v_t, cfg.stride_g_t,
     cfg.stride_beta_t) = [int(s) for s in strides]
    return cfg


@functools.lru_cache(maxsize=256)
def _config(num_heads, window, num_slots, record_slots, lower_bound, scale, strides, head_dim,
            record_format) -> KdaConfig:
    # the library only reads the config during the call, so one object per
    # distinct argument set serves every call
    return make_config(num_heads, window, num_slots, record_slots, lower_bound=lower_bound,
                       scale=scale, strides=strides, head_dim=head_dim,
                       record_format=record_format)


def kda_records_bytes(num_heads: int, window: int, record_slots: int) -> int:
    """Size in bytes of a raw-format records buffer (``kda_records_bytes``)."""
    return int(load_library().kda_records_bytes(num_heads, window, record_slots))


def kda_correction_records_bytes(num_heads: int, window: int, record_slots: int) -> int:
    """Size in bytes of a correction-format records buffer
    (``kda_correction_records_bytes``)."""
    return int(load_library().kda_correction_records_bytes(num_heads, window, record_slots))


@functools.lru_cache(maxsize=256)
def records_bytes(num_heads: int, window: int, record_slots: int, record_format: str) -> int:
    _format_code(record_format)
    fn = kda_records_bytes if record_format == "raw" else kda_correction_records_bytes
    return fn(num_heads, window, record_slots)


def allocate_records(num_heads: int, window: int, record_slots: int, device,
                     record_format: str = "raw") -> torch.Tensor:
    """A records buffer (raw or correction format) for ``record_slots``
    slots plus the scratch row, as a flat bf16 tensor."""
    nbytes = records_bytes(num_heads, window, record_slots, record_format)
    if nbytes == 0:
        raise ValueError("invalid record sizes")
    return torch.empty(nbytes // 2, dtype=torch.bfloat16, device=device)


def _check_records(records, H, window, record_slots, record_format):
    """The records buffer holds the format's size (sizes the library does
    not support are left for it to report)."""
    need = records_bytes(H, window, record_slots, record_format)
    if need > 0 and (records.numel() * records.element_size() < need
                     or not records.is_contiguous()):
        raise ValueError(f"records must be a contiguous buffer of at least {need} bytes "
                         f"for the {record_format} format")


def kda_verify(q, k, v, g_raw, beta_raw, A_log, g_bias, state_pool, cu_seqlens,
               state_indices, records, out, *, window: int, record_slots: int,
               lower_bound=None, scale=None, record_rows=None, pending=None,
               trajectory_out=None, error_word=None, record_format: str = "raw") -> torch.Tensor:
    """``kda_verify``: speculative verify from each row's checkpoint.

    q, k, v, g_raw: bf16 [T, H, 128] (token stride free, [H, D] packed);
    beta_raw: bf16 [T, H]; A_log fp32 [H]; g_bias fp32 [H*128];
    state_pool fp32 [S, H, 128, 128]; cu_seqlens int32 [B+1];
    state_indices int32 [B]; records: buffer from ``allocate_records``
    for the same ``record_format`` ("raw": k, v, g_raw and beta_raw per
    token; "correction": each token's fp32 delta with k and g_raw);
    out: bf16 [T, H, 128] contiguous.  Returns ``out``.
    """
    dev = state_pool.device
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    for name, t in (("q", q), ("k", k), ("v", v), ("g_raw", g_raw), ("beta_raw", beta_raw),
                    ("records", records), ("out", out)):
        _req(t, bf, name, dev)
    for name, t in (("A_log", A_log), ("g_bias", g_bias), ("state_pool", state_pool)):
        _req(t, f32, name, dev)
    _req(cu_seqlens, i32, "cu_seqlens", dev)
    _req(state_indices, i32, "state_indices", dev)
    _opt(record_rows, i32, "record_rows", dev)
    _opt(pending, i32, "pending", dev)
    _opt(trajectory_out, f32, "trajectory_out", dev)
    _opt(error_word, i32, "error_word", dev)
    S, H, D = _check_pool(state_pool)
    _check_gate(A_log, g_bias, H, D)
    for t in (cu_seqlens, state_indices):
        if not t.is_contiguous():
            raise ValueError("metadata tensors must be contiguous")
    B = state_indices.shape[0]
    if cu_seqlens.shape[0] != B + 1:
        raise ValueError("cu_seqlens must have B + 1 entries")
    _check_rows(B, record_slots, record_rows, pending, None, error_word)
    T = _tokens(q, "q", H, D)
    for name, t in (("k", k), ("v", v), ("g_raw", g_raw), ("out", out)):
        if _tokens(t, name, H, D) != T:
            raise ValueError(f"{name} has a different token count from q")
    if _tokens(beta_raw, "beta_raw", H, None) != T:
        raise ValueError("beta_raw has a different token count from q")
    if not out.is_contiguous():
        raise ValueError("out must be contiguous")
    if trajectory_out is not None:
        if not trajectory_out.is_contiguous():
            raise ValueError("trajectory_out must be contiguous")
        _at_least(trajectory_out, T * H * D * D, "trajectory_out")
    strides = (_token_stride(q), _token_stride(k), _token_stride(v), _token_stride(g_raw),
               _token_stride(beta_raw))
    cfg = _config(H, window, S, record_slots, lower_bound, scale, strides, state_pool.shape[-1],
                  record_format)
    _check_records(records, H, window, record_slots, record_format)
    lib = load_library()
    st = lib.kda_verify(ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(v), _ptr(g_raw),
                        _ptr(beta_raw), _ptr(A_log), _ptr(g_bias), _ptr(state_pool),
                        _ptr(cu_seqlens), _ptr(state_indices), B, _ptr(record_rows),
                        _ptr(pending), _ptr(records), _ptr(out), _ptr(trajectory_out),
                        _ptr(error_word), _stream_ptr(dev))
    _check("kda_verify", st)
    return out


def kda_commit(A_log, g_bias, state_pool, cu_seqlens, state_indices, num_accepted, records,
               *, window: int, record_slots: int, lower_bound=None, record_rows=None,
               pending=None, eager=None, error_word=None, record_format: str = "raw") -> None:
    """``kda_commit``: fold each row's accepted tokens into its checkpoint
    (eager), or store them as pending replays (deferred, ``pending`` given).
    ``record_format`` must be the one the verify wrote ``records`` with."""
    dev = state_pool.device
    f32, i32 = torch.float32, torch.int32
    for name, t in (("A_log", A_log), ("g_bias", g_bias), ("state_pool", state_pool)):
        _req(t, f32, name, dev)
    _req(records, torch.bfloat16, "records", dev)
    _req(cu_seqlens, i32, "cu_seqlens", dev)
    _req(state_indices, i32, "state_indices", dev)
    _req(num_accepted, i32, "num_accepted", dev)
    _opt(record_rows, i32, "record_rows", dev)
    _opt(pending, i32, "pending", dev)
    _opt(eager, torch.uint8, "eager", dev)
    _opt(error_word, i32, "error_word", dev)
    S, H, D = _check_pool(state_pool)
    _check_gate(A_log, g_bias, H, D)
    B = state_indices.shape[0]
    for t in (cu_seqlens, state_indices, num_accepted):
        if not t.is_contiguous():
            raise ValueError("metadata tensors must be contiguous")
    if cu_seqlens.shape[0] != B + 1 or num_accepted.shape[0] < B:
        raise ValueError("metadata sizes do not match the batch")
    _check_rows(B, record_slots, record_rows, pending, eager, error_word)
    cfg = _config(H, window, S, record_slots, lower_bound, None, (1, 1, 1, 1, 1), D,
                  record_format)
    _check_records(records, H, window, record_slots, record_format)
    lib = load_library()
    st = lib.kda_commit(ctypes.byref(cfg), _ptr(A_log), _ptr(g_bias), _ptr(state_pool),
                        _ptr(cu_seqlens), _ptr(state_indices), B, _ptr(num_accepted),
                        _ptr(record_rows), _ptr(records), _ptr(pending), _ptr(eager),
                        _ptr(error_word), _stream_ptr(dev))
    _check("kda_commit", st)


def kda_flush(A_log, g_bias, state_pool, state_indices, records, pending, *, window: int,
              record_slots: int, lower_bound=None, record_rows=None, error_word=None,
              record_format: str = "raw") -> None:
    """``kda_flush``: fold pending replays into the checkpoints in place
    (``record_format`` as for ``kda_commit``)."""
    dev = state_pool.device
    f32, i32 = torch.float32, torch.int32
    for name, t in (("A_log", A_log), ("g_bias", g_bias), ("state_pool", state_pool)):
        _req(t, f32, name, dev)
    _req(records, torch.bfloat16, "records", dev)
    _req(state_indices, i32, "state_indices", dev)
    _req(pending, i32, "pending", dev)
    _opt(record_rows, i32, "record_rows", dev)
    _opt(error_word, i32, "error_word", dev)
    S, H, D = _check_pool(state_pool)
    _check_gate(A_log, g_bias, H, D)
    B = state_indices.shape[0]
    if not state_indices.is_contiguous():
        raise ValueError("metadata tensors must be contiguous")
    _check_rows(B, record_slots, record_rows, pending, None, error_word)
    cfg = _config(H, window, S, record_slots, lower_bound, None, (1, 1, 1, 1, 1), D,
                  record_format)
    _check_records(records, H, window, record_slots, record_format)
    lib = load_library()
    st = lib.kda_flush(ctypes.byref(cfg), _ptr(A_log), _ptr(g_bias), _ptr(state_pool),
                       _ptr(state_indices), B, _ptr(record_rows), _ptr(records), _ptr(pending),
                       _ptr(error_word), _stream_ptr(dev))
    _check("kda_flush", st)


def make_conv_config(conv_state: torch.Tensor, window: int) -> KdaConvConfig:
    """``kda_conv_config`` of a conv-state pool viewed as [S, conv_dim, width]
    (any strides: a channel-major pool or a transposed view of a
    column-major one)."""
    if conv_state.dim() != 3:
        raise ValueError("conv_state must be viewed as [S, conv_dim, width]")
    cc = KdaConvConfig()
    cc.num_slots, cc.conv_dim, cc.width = (int(x) for x in conv_state.shape)
    cc.window = window
    cc.elem_bytes = conv_state.element_size()
    cc.reserved = 0
    cc.stride_slot, cc.stride_dim, cc.stride_col = (int(x) for x in conv_state.stride())
    return cc


def kda_conv_compact(conv_state, cu_seqlens, state_indices, num_accepted, *, window: int,
                     error_word=None) -> None:
    """``kda_conv_compact``: move each committed row's conv window (starting
    at column n - 1) to column 0, in place.  conv_state: [S, conv_dim, width]
    view of 2- or 4-byte elements."""
    dev = conv_state.device
    i32 = torch.int32
    if conv_state.element_size() not in (2, 4):
        raise TypeError("conv_state elements must be 2 or 4 bytes")
    _req(cu_seqlens, i32, "cu_seqlens", dev)
    _req(state_indices, i32, "state_indices", dev)
    _req(num_accepted, i32, "num_accepted", dev)
    _opt(error_word, i32, "error_word", dev)
    for t in (cu_seqlens, state_indices, num_accepted):
        if not t.is_contiguous():
            raise ValueError("metadata tensors must be contiguous")
    B = state_indices.shape[0]
    if cu_seqlens.shape[0] != B + 1 or num_accepted.shape[0] < B:
        raise ValueError("metadata sizes do not match the batch")
    cc = make_conv_config(conv_state, window)
    lib = load_library()
    st = lib.kda_conv_compact(ctypes.byref(cc), _ptr(conv_state), _ptr(cu_seqlens),
                              _ptr(state_indices), B, _ptr(num_accepted), _ptr(error_word),
                              _stream_ptr(dev))
    _check("kda_conv_compact", st)


def make_align(block_table, num_computed, block_size: int, request_indices=None) -> KdaAlign:
    """``kda_align`` of an int32 block table [num_requests, width] (row stride
    free, columns contiguous) and int32 num_computed [num_requests]."""
    if block_table.dim() != 2 or block_table.stride(1) != 1:
        raise ValueError("block_table must be [num_requests, width] with contiguous columns")
    al = KdaAlign()
    al.block_table = block_table.data_ptr()
    al.block_table_stride = block_table.stride(0)
    al.block_table_width = block_table.shape[1]
    al.block_size = block_size
    al.num_requests = block_table.shape[0]
    al.reserved = 0
    al.num_computed = num_computed.data_ptr()
    al.request_indices = None if request_indices is None else request_indices.data_ptr()
    return al


def _check_align(block_table, num_computed, request_indices, dev):
    i32 = torch.int32
    _req(block_table, i32, "block_table", dev)
    _req(num_computed, i32, "num_computed", dev)
    _opt(request_indices, i32, "request_indices", dev)
    if num_computed.shape[0] < block_table.shape[0] or not num_computed.is_contiguous():
        raise ValueError("num_computed must be contiguous with one entry per request")
    if request_indices is not None and not request_indices.is_contiguous():
        raise ValueError("request_indices must be contiguous")


def kda_commit_align(A_log, g_bias, state_pool, cu_seqlens, state_indices, num_accepted, records,
                     block_table, num_computed, *, block_size: int, window: int,
                     record_slots: int, lower_bound=None, record_rows=None,
                     request_indices=None, pending=None, eager=None, error_word=None,
                     record_format: str = "raw") -> None:
    """``kda_commit_align``: the commit writing the final and boundary blocks
    of a paged state cache.  num_accepted, num_computed and the block table
    rows are per request; ``record_format`` as for ``kda_commit``.  With
    ``pending`` (and optionally ``eager``), the deferred form: rows that stay
    in their own slot and owe no boundary block only record their pending
    replay."""
    dev = state_pool.device
    f32, i32 = torch.float32, torch.int32
    for name, t in (("A_log", A_log), ("g_bias", g_bias), ("state_pool", state_pool)):
        _req(t, f32, name, dev)
    _req(records, torch.bfloat16, "records", dev)
    _req(cu_seqlens, i32, "cu_seqlens", dev)
    _req(state_indices, i32, "state_indices", dev)
    _req(num_accepted, i32, "num_accepted", dev)
    _opt(record_rows, i32, "record_rows", dev)
    _opt(pending, i32, "pending", dev)
    _opt(eager, torch.uint8, "eager", dev)
    _opt(error_word, i32, "error_word", dev)
    _check_align(block_table, num_computed, request_indices, dev)
    S, H, D = _check_pool(state_pool)
    _check_gate(A_log, g_bias, H, D)
    B = state_indices.shape[0]
    for t in (cu_seqlens, state_indices, num_accepted):
        if not t.is_contiguous():
            raise ValueError("metadata tensors must be contiguous")
    if cu_seqlens.shape[0] != B + 1 or num_accepted.shape[0] < block_table.shape[0]:
        raise ValueError("metadata sizes do not match the batch")
    _check_rows(B, record_slots, record_rows, pending, eager, error_word)
    if request_indices is not None:
        _at_least(request_indices, B, "request_indices")
    cfg = _config(H, window, S, record_slots, lower_bound, None, (1, 1, 1, 1, 1), D,
                  record_format)
    _check_records(records, H, window, record_slots, record_format)
    al = make_align(block_table, num_computed, block_size, request_indices)
    lib = load_library()
    st = lib.kda_commit_align(ctypes.byref(cfg), _ptr(A_log), _ptr(g_bias), _ptr(state_pool),
                              _ptr(cu_seqlens), _ptr(state_indices), B, _ptr(num_accepted),
                              _ptr(record_rows), _ptr(records), ctypes.byref(al),
                              _ptr(pending), _ptr(eager), _ptr(error_word), _stream_ptr(dev))
    _check("kda_commit_align", st)


def kda_conv_compact_align(conv_state, cu_seqlens, state_indices, num_accepted, block_table,
                           num_computed, *, block_size: int, window: int,
                           request_indices=None, error_word=None) -> None:
    """``kda_conv_compact_align``: the conv windows of each committed row go
    to its final and boundary blocks."""
    dev = conv_state.device
    i32 = torch.int32
    if conv_state.element_size() not in (2, 4):
        raise TypeError("conv_state elements must be 2 or 4 bytes")
    _req(cu_seqlens, i32, "cu_seqlens", dev)
    _req(state_indices, i32, "state_indices", dev)
    _req(num_accepted, i32, "num_accepted", dev)
    _opt(error_word, i32, "error_word", dev)
    _check_align(block_table, num_computed, request_indices, dev)
    B = state_indices.shape[0]
    if cu_seqlens.shape[0] != B + 1 or num_accepted.shape[0] < block_table.shape[0]:
        raise ValueError("metadata sizes do not match the batch")
    cc = make_conv_config(conv_state, window)
    al = make_align(block_table, num_computed, block_size, request_indices)
    lib = load_library()
    st = lib.kda_conv_compact_align(ctypes.byref(cc), _ptr(conv_state), _ptr(cu_seqlens),
                                    _ptr(state_indices), B, _ptr(num_accepted),
                                    ctypes.byref(al), _ptr(error_word), _stream_ptr(dev))
    _check("kda_conv_compact_align", st)


def kda_record_state_blocks(idx_mapping, num_sampled, num_computed, state_column, num_accepted,
                            *, block_size: int, block_table_width: int, num_rows=None,
                            request_indices=None, error_word=None) -> None:
    """``kda_record_state_blocks``: after an align-mode commit, point each
    committed request's running state column at the block of its last
    committed token and reset its accepted count to 1.  idx_mapping,
    num_sampled and num_computed are int32 per request; state_column and
    num_accepted int32 per running slot.  ``num_rows`` spec rows (default:
    request_indices' length, else one per request)."""
    dev = state_column.device
    i32 = torch.int32
    for name, t in (("idx_mapping", idx_mapping), ("num_sampled", num_sampled),
                    ("num_computed", num_computed), ("state_column", state_column),
                    ("num_accepted", num_accepted)):
        _req(t, i32, name, dev)
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    _opt(request_indices, i32, "request_indices", dev)
    _opt(error_word, i32, "error_word", dev)
    num_requests = idx_mapping.shape[0]
    if num_sampled.shape[0] < num_requests or num_computed.shape[0] < num_requests:
        raise ValueError("num_sampled and num_computed need one entry per request")
    if num_accepted.shape[0] != state_column.shape[0]:
        raise ValueError("state_column and num_accepted must have the same length")
    if num_rows is None:
        num_rows = num_requests if request_indices is None else request_indices.shape[0]
    if request_indices is not None:
        if not request_indices.is_contiguous():
            raise ValueError("request_indices must be contiguous")
        _at_least(request_indices, num_rows, "request_indices")
    elif num_rows > num_requests:
        raise ValueError("more spec rows than requests without request_indices")
    al = KdaAlign()
    al.block_table = None  # not read by this call
    al.block_table_stride = 0
    al.block_table_width = block_table_width
    al.block_size = block_size
    al.num_requests = num_requests
    al.reserved = 0
    al.num_computed = num_computed.data_ptr()
    al.request_indices = None if request_indices is None else request_indices.data_ptr()
    lib = load_library()
    st = lib.kda_record_state_blocks(ctypes.byref(al), _ptr(idx_mapping), _ptr(num_sampled),
                                     num_rows, _ptr(state_column), _ptr(num_accepted),
                                     state_column.shape[0], _ptr(error_word), _stream_ptr(dev))
    _check("kda_record_state_blocks", st)
