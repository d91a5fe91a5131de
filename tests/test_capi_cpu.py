"""CPU checks of the C ABI: the library builds, loads, exports every entry
point ``include/kda.h`` declares, and its host-side argument checks return
the documented status codes.  No case here reaches a kernel launch: each one
fails a host check (or has B == 0), so nothing touches a GPU."""

import ctypes
import os
import re

import pytest

from linear_attention_speculative_kda_gb300 import api
from linear_attention_speculative_kda_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return api.load_library()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert set(names) == set(api.EXPORTED)
    for name in names:
        assert hasattr(lib, name), name
    assert lib.kda_abi_version() == 4
    assert lib.kda_status_string(api.KDA_ERR_CUDA) == b"KDA_ERR_CUDA"


def test_records_bytes(lib):
    assert api.kda_records_bytes(16, 4, 1024) == 1025 * 16 * 4 * 392 * 2
    assert api.kda_records_bytes(1, 8, 0) == 1 * 8 * 392 * 2
    assert api.kda_records_bytes(0, 4, 4) == 0
    assert api.kda_records_bytes(4, 9, 4) == 0
    assert api.kda_records_bytes(4, 4, -1) == 0


def test_correction_records_bytes(lib):
    # fp32 delta + bf16 k + bf16 g_raw = 1024 bytes per token, scratch row included
    assert api.kda_correction_records_bytes(16, 4, 1024) == 1025 * 16 * 4 * 1024
    assert api.kda_correction_records_bytes(1, 8, 0) == 8 * 1024
    assert api.kda_correction_records_bytes(0, 4, 4) == 0
    assert api.kda_correction_records_bytes(4, 9, 4) == 0
    assert api.records_bytes(2, 4, 3, "correction") == 4 * 2 * 4 * 1024
    assert api.records_bytes(2, 4, 3, "raw") == api.kda_records_bytes(2, 4, 3)
    with pytest.raises(ValueError):
        api.records_bytes(2, 4, 3, "fp8")


def test_record_format_host_checks(lib):
    cfg = _cfg()
    cfg.record_format = 2
    assert _verify(lib, cfg) == api.KDA_ERR_INVALID_ARG
    cfg = _cfg()
    cfg.reserved = 1
    assert _verify(lib, cfg) == api.KDA_ERR_INVALID_ARG
    cfg = _cfg()
    cfg.record_format = 1
    c = ctypes.byref(cfg)
    assert _verify(lib, cfg, q=None) == api.KDA_ERR_INVALID_ARG   # format fine, pointer not
    assert lib.kda_flush(c, FAKE, FAKE, FAKE, FAKE, 3, None, FAKE, None, None,
                         None) == api.KDA_ERR_INVALID_ARG
    bad = _cfg()
    bad.record_format = -1
    assert lib.kda_commit(ctypes.byref(bad), FAKE, FAKE, FAKE, FAKE, FAKE, 3, FAKE, None, FAKE,
                          None, None, None, None) == api.KDA_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        api.make_config(2, 4, 8, 4, record_format="fp16")


FAKE = 0x100000  # an aligned address that is never dereferenced


def _cfg(**kw):
    base = dict(num_heads=2, window=4, num_slots=8, record_slots=4, lower_bound=None,
                strides=(3 * 2 * 128, 3 * 2 * 128, 3 * 2 * 128, 2 * 128, 10))
    base.update(kw)
    return api.make_config(base["num_heads"], base["window"], base["num_slots"],
                           base["record_slots"], lower_bound=base["lower_bound"],
                           strides=base["strides"], head_dim=base.get("head_dim", 128))


def _verify(lib, cfg, B=3, **ptrs):
    p = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, a_log=FAKE, g_bias=FAKE, pool=FAKE,
             cu=FAKE, slots=FAKE, rr=None, pending=None, records=FAKE, out=FAKE, traj=None,
             err=None)
    p.update(ptrs)
    cfgp = None if cfg is None else ctypes.byref(cfg)
    return lib.kda_verify(cfgp, p["q"], p["k"], p["v"], p["g"], p["beta"], p["a_log"],
                          p["g_bias"], p["pool"], p["cu"], p["slots"], B, p["rr"],
                          p["pending"], p["records"], p["out"], p["traj"], p["err"], None)


def test_verify_host_checks(lib):
    assert _verify(lib, None) == api.KDA_ERR_INVALID_ARG
    assert _verify(lib, _cfg(head_dim=64)) == api.KDA_ERR_UNSUPPORTED
    assert _verify(lib, _cfg(window=9)) == api.KDA_ERR_UNSUPPORTED
    assert _verify(lib, _cfg(num_heads=32768)) == api.KDA_ERR_UNSUPPORTED
    assert _verify(lib, _cfg(window=0)) == api.KDA_ERR_INVALID_ARG
    assert _verify(lib, _cfg(num_heads=0)) == api.KDA_ERR_INVALID_ARG
    assert _verify(lib, _cfg(), B=-1) == api.KDA_ERR_INVALID_ARG
    assert _verify(lib, _cfg(), q=None) == api.KDA_ERR_INVALID_ARG
    assert _verify(lib, _cfg(), out=None) == api.KDA_ERR_INVALID_ARG
    assert _verify(lib, _cfg(), q=FAKE + 2) == api.KDA_ERR_INVALID_ARG       # not 8-byte aligned
    assert _verify(lib, _cfg(), pool=FAKE + 4) == api.KDA_ERR_INVALID_ARG    # not 16-byte aligned
    assert _verify(lib, _cfg(), traj=FAKE + 8) == api.KDA_ERR_INVALID_ARG
    assert _verify(lib, _cfg(strides=(770, 768, 768, 256, 1))) == api.KDA_ERR_INVALID_ARG
    assert _verify(lib, _cfg(strides=(768, 768, 768, 256, 0))) == api.KDA_ERR_INVALID_ARG
    assert _verify(lib, _cfg(lower_bound=0.5)) == api.KDA_ERR_INVALID_ARG
    assert _verify(lib, _cfg(lower_bound=float("-inf"))) == api.KDA_ERR_INVALID_ARG
    assert _verify(lib, _cfg(record_slots=2), B=3) == api.KDA_ERR_INVALID_ARG  # B > R, no rr
    # nothing to do: OK without any launch, pointers not inspected
    assert _verify(lib, _cfg(), B=0) == api.KDA_OK
    assert _verify(lib, _cfg(), B=0, q=None, slots=None, cu=None) == api.KDA_OK
    assert _verify(lib, _cfg(window=9), B=0) == api.KDA_ERR_UNSUPPORTED


def test_commit_and_flush_host_checks(lib):
    cfg = _cfg()
    c = ctypes.byref(cfg)
    # eager mask without pending is meaningless
    assert lib.kda_commit(c, FAKE, FAKE, FAKE, FAKE, FAKE, 3, FAKE, None, FAKE, None, FAKE,
                          None, None) == api.KDA_ERR_INVALID_ARG
    assert lib.kda_commit(c, FAKE, FAKE, FAKE, FAKE, FAKE, 3, None, None, FAKE, None, None,
                          None, None) == api.KDA_ERR_INVALID_ARG
    assert lib.kda_commit(c, FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE, None, FAKE, None, None,
                          None, None) == api.KDA_OK
    assert lib.kda_flush(c, FAKE, FAKE, FAKE, FAKE, 3, None, FAKE, None, None,
                         None) == api.KDA_ERR_INVALID_ARG
    assert lib.kda_flush(c, FAKE, FAKE, FAKE, FAKE, 0, None, FAKE, FAKE, None,
                         None) == api.KDA_OK


def _conv(lib, B=3, cc=None, conv=FAKE, cu=FAKE, slots=FAKE, acc=FAKE, err=None, **kw):
    if cc is None:
        base = dict(num_slots=8, conv_dim=384, width=6, window=4, elem_bytes=2, reserved=0,
                    stride_slot=384 * 6, stride_dim=6, stride_col=1)
        base.update(kw)
        cc = api.KdaConvConfig(**base)
    ccp = None if cc is False else ctypes.byref(cc)
    return lib.kda_conv_compact(ccp, conv, cu, slots, B, acc, err, None)


def test_conv_compact_host_checks(lib):
    assert _conv(lib, cc=False) == api.KDA_ERR_INVALID_ARG
    assert _conv(lib, elem_bytes=8) == api.KDA_ERR_INVALID_ARG
    assert _conv(lib, width=3) == api.KDA_ERR_INVALID_ARG            # narrower than the window
    assert _conv(lib, width=20) == api.KDA_ERR_UNSUPPORTED           # history 17 > 16
    assert _conv(lib, window=9, width=12) == api.KDA_ERR_UNSUPPORTED
    assert _conv(lib, window=0) == api.KDA_ERR_INVALID_ARG
    assert _conv(lib, conv_dim=0) == api.KDA_ERR_INVALID_ARG
    assert _conv(lib, stride_col=0) == api.KDA_ERR_INVALID_ARG
    assert _conv(lib, reserved=1) == api.KDA_ERR_INVALID_ARG
    assert _conv(lib, B=-1) == api.KDA_ERR_INVALID_ARG
    assert _conv(lib, conv=None) == api.KDA_ERR_INVALID_ARG
    assert _conv(lib, acc=None) == api.KDA_ERR_INVALID_ARG
    assert _conv(lib, conv=FAKE + 1) == api.KDA_ERR_INVALID_ARG      # not element-aligned
    assert _conv(lib, elem_bytes=4, conv=FAKE + 2) == api.KDA_ERR_INVALID_ARG
    assert _conv(lib, cu=FAKE + 2) == api.KDA_ERR_INVALID_ARG
    # B == 0: nothing to do, and no pointer is looked at
    assert _conv(lib, B=0, conv=None, cu=None, slots=None, acc=None) == api.KDA_OK


def _align(**kw):
    base = dict(block_table=FAKE, block_table_stride=8, block_table_width=8, block_size=16,
                num_requests=4, reserved=0, num_computed=FAKE, request_indices=None)
    base.update(kw)
    return api.KdaAlign(**base)


def _commit_align(lib, al, cfg=None, B=3, **ptrs):
    p = dict(a_log=FAKE, g_bias=FAKE, pool=FAKE, cu=FAKE, slots=FAKE, acc=FAKE, rr=None,
             records=FAKE, pending=None, eager=None, err=None)
    p.update(ptrs)
    cfg = _cfg() if cfg is None else cfg
    alp = None if al is None else ctypes.byref(al)
    return lib.kda_commit_align(ctypes.byref(cfg), p["a_log"], p["g_bias"], p["pool"], p["cu"],
                                p["slots"], B, p["acc"], p["rr"], p["records"], alp,
                                p["pending"], p["eager"], p["err"], None)


def test_commit_align_host_checks(lib):
    assert _commit_align(lib, None) == api.KDA_ERR_INVALID_ARG
    assert _commit_align(lib, _align(block_table=None)) == api.KDA_ERR_INVALID_ARG
    assert _commit_align(lib, _align(num_computed=None)) == api.KDA_ERR_INVALID_ARG
    assert _commit_align(lib, _align(block_size=3)) == api.KDA_ERR_INVALID_ARG   # < window 4
    assert _commit_align(lib, _align(block_table_width=0)) == api.KDA_ERR_INVALID_ARG
    assert _commit_align(lib, _align(block_table_stride=4)) == api.KDA_ERR_INVALID_ARG
    assert _commit_align(lib, _align(num_requests=0)) == api.KDA_ERR_INVALID_ARG
    assert _commit_align(lib, _align(reserved=1)) == api.KDA_ERR_INVALID_ARG
    assert _commit_align(lib, _align(block_table=FAKE + 2)) == api.KDA_ERR_INVALID_ARG
    assert _commit_align(lib, _align(request_indices=FAKE + 1)) == api.KDA_ERR_INVALID_ARG
    assert _commit_align(lib, _align(), acc=None) == api.KDA_ERR_INVALID_ARG
    assert _commit_align(lib, _align(), cfg=_cfg(window=9)) == api.KDA_ERR_UNSUPPORTED
    assert _commit_align(lib, _align(), B=-1) == api.KDA_ERR_INVALID_ARG
    assert _commit_align(lib, None, B=0) == api.KDA_OK
    # the deferred form: an eager mask needs pending; pending needs 4-byte alignment
    assert _commit_align(lib, _align(), eager=FAKE) == api.KDA_ERR_INVALID_ARG
    assert _commit_align(lib, _align(), pending=FAKE + 2) == api.KDA_ERR_INVALID_ARG


def test_conv_compact_align_host_checks(lib):
    cc = api.KdaConvConfig(num_slots=8, conv_dim=64, width=6, window=4, elem_bytes=2, reserved=0,
                           stride_slot=64 * 6, stride_dim=6, stride_col=1)

    def call(al, B=3, cc=cc):
        alp = None if al is None else ctypes.byref(al)
        return lib.kda_conv_compact_align(ctypes.byref(cc), FAKE, FAKE, FAKE, B, FAKE, alp, None,
                                          None)

    assert call(None) == api.KDA_ERR_INVALID_ARG
    assert call(_align(block_size=2)) == api.KDA_ERR_INVALID_ARG
    assert call(_align(num_computed=None)) == api.KDA_ERR_INVALID_ARG
    assert call(_align(), B=-1) == api.KDA_ERR_INVALID_ARG
    assert call(None, B=0) == api.KDA_OK


def test_record_state_blocks_host_checks(lib):
    def call(al, B=3, idx=FAKE, ns=FAKE, col=FAKE, acc=FAKE, num_states=8, err=None):
        alp = None if al is None else ctypes.byref(al)
        return lib.kda_record_state_blocks(alp, idx, ns, B, col, acc, num_states, err, None)

    assert call(None) == api.KDA_ERR_INVALID_ARG
    assert call(_align(block_size=0)) == api.KDA_ERR_INVALID_ARG
    assert call(_align(block_table_width=0)) == api.KDA_ERR_INVALID_ARG
    assert call(_align(num_requests=0)) == api.KDA_ERR_INVALID_ARG
    assert call(_align(reserved=1)) == api.KDA_ERR_INVALID_ARG
    assert call(_align(num_computed=None)) == api.KDA_ERR_INVALID_ARG
    assert call(_align(num_computed=FAKE + 2)) == api.KDA_ERR_INVALID_ARG
    assert call(_align(request_indices=FAKE + 1)) == api.KDA_ERR_INVALID_ARG
    assert call(_align(), idx=None) == api.KDA_ERR_INVALID_ARG
    assert call(_align(), ns=None) == api.KDA_ERR_INVALID_ARG
    assert call(_align(), col=FAKE + 2) == api.KDA_ERR_INVALID_ARG
    assert call(_align(), acc=None) == api.KDA_ERR_INVALID_ARG
    assert call(_align(), err=FAKE + 1) == api.KDA_ERR_INVALID_ARG
    assert call(_align(), num_states=0) == api.KDA_ERR_INVALID_ARG
    assert call(_align(), B=-1) == api.KDA_ERR_INVALID_ARG
    # B == 0: nothing to do, and no pointer is looked at
    assert call(None, B=0, idx=None, ns=None, col=None, acc=None) == api.KDA_OK


def test_binding_refuses_small_records_buffer(lib):
    # the size check runs before any device call, so CPU tensors suffice
    import torch
    T, H = 4, 2
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    act = torch.zeros((T, H, 128), dtype=bf)
    pool = torch.zeros((3, H, 128, 128), dtype=f32)
    raw = torch.zeros(api.kda_records_bytes(H, 4, 1) // 2, dtype=bf)
    args = (act, act, act, act, torch.zeros((T, H), dtype=bf), torch.zeros(H, dtype=f32),
            torch.zeros(H * 128, dtype=f32), pool, torch.tensor([0, 4], dtype=i32),
            torch.tensor([1], dtype=i32))
    with pytest.raises(ValueError, match="correction"):
        api.kda_verify(*args, raw, torch.zeros_like(act), window=4, record_slots=1,
                       record_format="correction")
    with pytest.raises(ValueError, match="raw"):
        api.kda_verify(*args, raw[:-1], torch.zeros_like(act), window=4, record_slots=1)
    with pytest.raises(ValueError):
        api.kda_commit(torch.zeros(H, dtype=f32), torch.zeros(H * 128, dtype=f32), pool,
                       torch.tensor([0, 4], dtype=i32), torch.tensor([1], dtype=i32),
                       torch.tensor([2], dtype=i32), raw, window=4, record_slots=1,
                       record_format="correction")


def test_error_word_alignment(lib):
    # the kernels OR bits into the error word with a 32-bit atomic: a pointer
    # off a 4-byte boundary is refused before anything is launched
    c = ctypes.byref(_cfg())
    assert _verify(lib, _cfg(), err=FAKE + 2) == api.KDA_ERR_INVALID_ARG
    assert lib.kda_commit(c, FAKE, FAKE, FAKE, FAKE, FAKE, 3, FAKE, None, FAKE, None, None,
                          FAKE + 1, None) == api.KDA_ERR_INVALID_ARG
    assert lib.kda_flush(c, FAKE, FAKE, FAKE, FAKE, 3, None, FAKE, FAKE, FAKE + 2,
                         None) == api.KDA_ERR_INVALID_ARG
    assert _commit_align(lib, _align(), err=FAKE + 2) == api.KDA_ERR_INVALID_ARG
    assert _conv(lib, err=FAKE + 2) == api.KDA_ERR_INVALID_ARG


def _host_args(T=4, H=2, S=3, B=1, R=1):
    """Consistent CPU tensors for the binding's checks (never launched: each
    test below breaks one of them, and the check raises first)."""
    import torch
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    return dict(
        q=torch.zeros((T, H, 128), dtype=bf), k=torch.zeros((T, H, 128), dtype=bf),
        v=torch.zeros((T, H, 128), dtype=bf), g_raw=torch.zeros((T, H, 128), dtype=bf),
        beta_raw=torch.zeros((T, H), dtype=bf), A_log=torch.zeros(H, dtype=f32),
        g_bias=torch.zeros(H * 128, dtype=f32), state_pool=torch.zeros((S, H, 128, 128), dtype=f32),
        cu_seqlens=torch.tensor([0, T], dtype=i32), state_indices=torch.tensor([1], dtype=i32),
        records=torch.zeros(api.kda_records_bytes(H, 4, R) // 2, dtype=bf),
        out=torch.zeros((T, H, 128), dtype=bf))


def _bad_verify(**change):
    a = _host_args()
    kw = dict(window=4, record_slots=1)
    for name, val in change.items():
        (a if name in a else kw)[name] = val
    with pytest.raises(ValueError):
        api.kda_verify(a["q"], a["k"], a["v"], a["g_raw"], a["beta_raw"], a["A_log"], a["g_bias"],
                       a["state_pool"], a["cu_seqlens"], a["state_indices"], a["records"],
                       a["out"], **kw)


def test_binding_checks_shapes_before_any_launch(lib):
    import torch
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    _bad_verify(k=torch.zeros((4, 1, 128), dtype=bf))            # fewer heads than the pool
    _bad_verify(v=torch.zeros((4, 2, 64), dtype=bf))             # not 128 channels
    _bad_verify(g_raw=torch.zeros((3, 2, 128), dtype=bf))        # another token count
    _bad_verify(beta_raw=torch.zeros((4, 1), dtype=bf))          # beta needs H columns
    _bad_verify(out=torch.zeros((2, 2, 128), dtype=bf))          # out shorter than q
    _bad_verify(q=torch.zeros((2, 4, 2, 128), dtype=bf))         # a batch dimension > 1
    _bad_verify(A_log=torch.zeros(1, dtype=f32))                 # fewer than H entries
    _bad_verify(g_bias=torch.zeros(128, dtype=f32))              # fewer than H * 128
    _bad_verify(state_pool=torch.zeros((3, 2, 128, 64), dtype=f32))
    _bad_verify(pending=torch.zeros(0, dtype=i32))               # fewer than record_slots
    _bad_verify(record_rows=torch.zeros(0, dtype=i32))           # fewer than B
    _bad_verify(error_word=torch.zeros(0, dtype=i32))
    _bad_verify(trajectory_out=torch.zeros(4 * 2 * 128 * 127, dtype=f32))
    a = _host_args()
    common = (a["A_log"], a["g_bias"], a["state_pool"], a["cu_seqlens"], a["state_indices"])
    with pytest.raises(ValueError):   # eager mask shorter than the batch
        api.kda_commit(*common, torch.tensor([2], dtype=i32), a["records"], window=4,
                       record_slots=1, pending=torch.zeros(1, dtype=i32),
                       eager=torch.zeros(0, dtype=torch.uint8))
    with pytest.raises(ValueError):   # g_bias of one head for a two-head pool
        api.kda_commit(a["A_log"], torch.zeros(128, dtype=f32), *common[2:],
                       torch.tensor([2], dtype=i32), a["records"], window=4, record_slots=1)
    with pytest.raises(ValueError):   # pending shorter than the record slots
        api.kda_flush(a["A_log"], a["g_bias"], a["state_pool"], a["state_indices"], a["records"],
                      torch.zeros(0, dtype=i32), window=4, record_slots=1)


def test_binding_checks_record_state_blocks_sizes(lib):
    # every check raises before the library is called, so CPU tensors suffice
    import torch
    i32 = torch.int32
    idx = torch.zeros(4, dtype=i32)
    col = torch.zeros(6, dtype=i32)

    def call(**kw):
        args = dict(idx_mapping=idx, num_sampled=torch.zeros(4, dtype=i32),
                    num_computed=torch.zeros(4, dtype=i32), state_column=col,
                    num_accepted=torch.zeros(6, dtype=i32))
        args.update(kw)
        api.kda_record_state_blocks(block_size=16, block_table_width=4, **args)

    with pytest.raises(ValueError, match="per request"):
        call(num_sampled=torch.zeros(3, dtype=i32))
    with pytest.raises(ValueError, match="same length"):
        call(num_accepted=torch.zeros(5, dtype=i32))
    with pytest.raises(ValueError, match="more spec rows"):
        call(num_rows=5)
    with pytest.raises(ValueError, match="request_indices needs"):
        call(request_indices=torch.zeros(2, dtype=i32), num_rows=3)
    with pytest.raises(TypeError):
        call(idx_mapping=torch.zeros(4, dtype=torch.int64))
