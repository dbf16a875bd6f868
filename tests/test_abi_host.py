"""Host-side checks of the C ABI (no GPU needed, no compute calls).

The library must load, export every function include/sms.h declares, and
reject bad arguments on the host before any launch.  Pointer arguments here
are fake addresses: every call is rejected by validation before anything is
dereferenced or launched.
"""
import os
import re

import pytest
import torch

import scaled_masked_softmax_gb300 as sms
from scaled_masked_softmax_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sms.h")
INVALID, UNSUPPORTED = binding.SMS_ERR_INVALID_ARG, binding.SMS_ERR_UNSUPPORTED


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sms_\w+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    lib = binding.lib()
    names = _declared()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), f"libsms.so does not export {n}"
    assert set(names) == set(binding.SIGNATURES), "binding signatures out of sync with include/sms.h"
    assert sms.sms_version() == 100


def _fwd(**kw):
    a = dict(x=0x10000, mask=None, mask_numel=0, sb=0, sh=0, heads=1, y=0x20000, rows=4, cols=8, scale=1.0,
             causal=0, dtype=0, stream=None)
    a.update(kw)
    return binding.lib().sms_forward(a["x"], a["mask"], a["mask_numel"], a["sb"], a["sh"], a["heads"], a["y"],
                                     a["rows"], a["cols"], a["scale"], a["causal"], a["dtype"], a["stream"])


def _bwd(**kw):
    a = dict(y=0x10000, dy=0x20000, dx=0x30000, rows=4, cols=8, scale=1.0, causal=0, dtype=0, stream=None)
    a.update(kw)
    return binding.lib().sms_backward(a["y"], a["dy"], a["dx"], a["rows"], a["cols"], a["scale"], a["causal"],
                                      a["dtype"], a["stream"])


@pytest.mark.parametrize("kw", [
    dict(x=None), dict(y=None), dict(dtype=3), dict(dtype=-1), dict(rows=-1), dict(cols=0), dict(cols=-5),
    dict(cols=(1 << 30) + 1), dict(rows=1 << 40, cols=1 << 30), dict(scale=float("inf")), dict(scale=float("nan")),
    dict(x=0x10004), dict(y=0x20008), dict(y=0x10010),  # misaligned, partial overlap of y and x
    dict(mask=0x40000, mask_numel=8 * 8 - 1, cols=8, rows=8),  # [S,S] mask one element short
    dict(mask=0x40000, mask_numel=64, heads=0), dict(mask=0x40000, mask_numel=64, sb=-1),
    dict(mask=0x40004, mask_numel=64),  # misaligned mask
    dict(mask=0x40000, mask_numel=64, rows=16, cols=8, sb=64, heads=1),  # 2 batches, extent 128 > 64
    dict(mask=0x1ffe0, mask_numel=64, rows=8, cols=8),  # y overlaps the mask
])
def test_forward_rejects_bad_arguments(kw):
    assert _fwd(**kw) == INVALID
    assert binding.sms_last_error() != ""


@pytest.mark.parametrize("kw", [
    dict(y=None), dict(dy=None), dict(dx=None), dict(dtype=7), dict(rows=-2), dict(cols=0),
    dict(scale=float("nan")), dict(dx=0x30008), dict(dx=0x10010), dict(dx=0x20010)])
def test_backward_rejects_bad_arguments(kw):
    assert _bwd(**kw) == INVALID


def test_rows_zero_is_a_noop_without_device():
    assert _fwd(rows=0) == binding.SMS_OK
    assert _bwd(rows=0) == binding.SMS_OK
    assert _fwd(rows=0, x=None, y=None) == binding.SMS_OK  # empty tensors have NULL data pointers
    assert _bwd(rows=0, y=None, dy=None, dx=None) == binding.SMS_OK
    assert _fwd(rows=0, cols=0) == INVALID


def test_in_place_aliasing_passes_validation():
    # y == x and dx == dy are allowed; without a GPU the call then fails at the
    # device query (SMS_ERR_CUDA), never at validation
    if torch.cuda.is_available():
        pytest.skip("host-only check")
    assert _fwd(y=0x10000) == binding.SMS_ERR_CUDA
    assert _bwd(dx=0x20000) == binding.SMS_ERR_CUDA


def test_mask_extent_rule_for_partial_heads():
    # rows = 1.5 heads of S=8 with a [B,H,S,S] mask: the extent is the last
    # row's offset + cols, not B*H*S*S
    if torch.cuda.is_available():
        pytest.skip("host-only check")
    S, Hh = 8, 2
    rows = 12  # head 0 full, head 1 rows 0..3
    need = 1 * S * S + 3 * S + S  # h=1, q=3
    assert _fwd(mask=0x40000, mask_numel=need - 1, rows=rows, cols=S, heads=Hh, sb=Hh * S * S, sh=S * S) == INVALID
    assert _fwd(mask=0x40000, mask_numel=need, rows=rows, cols=S, heads=Hh, sb=Hh * S * S, sh=S * S) == \
        binding.SMS_ERR_CUDA


def test_status_strings_and_forced_path():
    for st in range(4):
        assert sms.sms_status_string(st)
    prev = sms.sms_set_forced_path(sms.SMS_PATH_CTA)
    assert sms.sms_set_forced_path(sms.SMS_PATH_ONLINE) == sms.SMS_PATH_CTA
    assert sms.sms_set_forced_path(prev) == sms.SMS_PATH_ONLINE
    assert sms.sms_set_forced_path(sms.SMS_PATH_STREAM) == sms.SMS_PATH_AUTO
    assert sms.sms_set_forced_path(sms.SMS_PATH_AUTO) == sms.SMS_PATH_STREAM
    with pytest.raises(ValueError):
        sms.sms_set_forced_path(6)
    with pytest.raises(ValueError):
        sms.sms_set_forced_path(9)
    prev = sms.sms_set_grid_limit(3)
    assert sms.sms_set_grid_limit(prev) == 3
    with pytest.raises(ValueError):
        sms.sms_set_grid_limit(-1)


def test_dispatcher_thresholds():
    W, C, O, R = sms.SMS_PATH_WARP, sms.SMS_PATH_CTA, sms.SMS_PATH_ONLINE, sms.SMS_PATH_RING
    for dt in (0, 1, 2):
        sixteen = dt != 0
        S = sms.SMS_PATH_STREAM
        assert sms.sms_select_path(1000, 64, dt) == (W if sixteen else S)  # short fp32 rows: prefetching groups
        assert sms.sms_select_path(1000, 512, dt) == (W if sixteen else S)
        assert sms.sms_select_path(1000, 513, dt) == W
        assert sms.sms_select_path(1000, 64, dt, True) == W
        assert sms.sms_select_path(1000, 1024, dt) == W
        assert sms.sms_select_path(1000, 4096, dt) == W
        assert sms.sms_select_path(1000, 8192, dt) == W
        # aligned 16-bit forward rows stay register-resident up to 256 lanes x 8 vectors
        assert sms.sms_select_path(1000, 16384, dt) == (W if sixteen else C)
        assert sms.sms_select_path(1000, 10248, dt) == (W if sixteen else C)  # 16-bit: 1281 vectors, 256 x 6
        assert sms.sms_select_path(1000, 10249, dt) == C  # unaligned 16-bit rows stop at 256 x 5 vectors
        assert sms.sms_select_path(1000, 16392, dt) == O  # beyond the staged path's forward registers
        # backward: 16-bit rows too wide for registers go to the bulk-copy rings (up to 2048 vectors)
        assert sms.sms_select_path(1000, 8192, dt, True) == (W if sixteen else C)
        assert sms.sms_select_path(1000, 16384, dt, True) == (R if sixteen else C)
        assert sms.sms_select_path(1000, 16392, dt, True) == (C if sixteen else O)
        assert sms.sms_select_path(1000, 1 << 20, dt) == O
        assert sms.sms_select_path(1000, 1 << 20, dt, True) == O
    assert sms.sms_select_path(1, 0, 0) == -1


@pytest.mark.parametrize("x_shape,m_shape,want", [
    ((2, 3, 8, 8), (8, 8), (0, 0, 3)),
    ((2, 3, 8, 8), (2, 1, 8, 8), (64, 0, 3)),
    ((2, 3, 8, 8), (2, 3, 8, 8), (192, 64, 3)),
    ((2, 3, 8, 8), (1, 3, 8, 8), (0, 64, 3)),
    ((2, 3, 8, 8), (1, 1, 8, 8), (0, 0, 3)),
    ((3, 8, 8), (3, 8, 8), (0, 64, 3)),
    ((4, 2, 3, 8, 8), (4, 2, 1, 8, 8), (64, 0, 3)),
])
def test_mask_layout(x_shape, m_shape, want):
    assert sms.mask_layout(x_shape, m_shape) == want


@pytest.mark.parametrize("x_shape,m_shape", [((2, 3, 8, 8), (3, 1, 8, 8)), ((2, 3, 8, 8), (2, 2, 8, 8)),
                                             ((2, 3, 8, 8), (8, 7)), ((4, 2, 3, 8, 8), (4, 1, 1, 8, 8))])
def test_mask_layout_rejects(x_shape, m_shape):
    with pytest.raises(ValueError):
        sms.mask_layout(x_shape, m_shape)


def _fwd_len(**kw):
    a = dict(x=0x10000, lengths=0x50000, heads=1, y=0x20000, rows=16, cols=8, scale=1.0, causal=0, dtype=0,
             stream=None)
    a.update(kw)
    return binding.lib().sms_forward_lengths(a["x"], a["lengths"], a["heads"], a["y"], a["rows"], a["cols"],
                                             a["scale"], a["causal"], a["dtype"], a["stream"])


def _bwd_len(**kw):
    a = dict(y=0x10000, dy=0x20000, dx=0x30000, lengths=0x50000, heads=1, rows=16, cols=8, scale=1.0, causal=0,
             dtype=0, stream=None)
    a.update(kw)
    return binding.lib().sms_backward_lengths(a["y"], a["dy"], a["dx"], a["lengths"], a["heads"], a["rows"],
                                              a["cols"], a["scale"], a["causal"], a["dtype"], a["stream"])


@pytest.mark.parametrize("kw", [
    dict(lengths=None), dict(lengths=0x50002), dict(heads=0), dict(heads=-3), dict(heads=(1 << 31) + 1),
    dict(x=None), dict(dtype=5), dict(cols=0), dict(scale=float("nan")), dict(y=0x20004),
    dict(lengths=0x20000 + 4 * 8 * 16 - 4),  # the lengths array (2 batches) overlaps y
])
def test_forward_lengths_rejects_bad_arguments(kw):
    assert _fwd_len(**kw) == INVALID
    assert binding.sms_last_error().startswith("sms_forward_lengths")


@pytest.mark.parametrize("kw", [
    dict(lengths=None), dict(lengths=0x50001), dict(heads=0), dict(dx=None), dict(dx=0x10010),
    dict(lengths=0x30000 + 4),  # overlaps dx
])
def test_backward_lengths_rejects_bad_arguments(kw):
    assert _bwd_len(**kw) == INVALID
    assert binding.sms_last_error().startswith("sms_backward_lengths")


def test_lengths_entry_points_pass_validation():
    # valid arguments reach the device query (no GPU here: SMS_ERR_CUDA); rows = 0 is a no-op
    if torch.cuda.is_available():
        pytest.skip("host-only check")
    assert _fwd_len() == binding.SMS_ERR_CUDA
    assert _bwd_len(heads=2, causal=1) == binding.SMS_ERR_CUDA
    assert _fwd_len(rows=0) == binding.SMS_OK
    assert _bwd_len(rows=0) == binding.SMS_OK


def _fwd_bool(**kw):
    a = dict(x=0x10000, mask=0x40000, mask_numel=64, sb=0, sh=0, heads=1, y=0x20000, rows=8, cols=8, scale=1.0,
             causal=0, dtype=0, stream=None)
    a.update(kw)
    return binding.lib().sms_forward_bool(a["x"], a["mask"], a["mask_numel"], a["sb"], a["sh"], a["heads"], a["y"],
                                          a["rows"], a["cols"], a["scale"], a["causal"], a["dtype"], a["stream"])


@pytest.mark.parametrize("kw", [
    dict(mask=None), dict(x=None), dict(dtype=4), dict(cols=0), dict(scale=float("nan")), dict(heads=0),
    dict(mask=0x40008),  # misaligned mask
    dict(mask_numel=63),  # [S,S] byte mask one element short
    dict(mask_numel=64, rows=16, sb=64),  # 2 batches reach byte 127
    dict(mask=0x1fff0, mask_numel=64),  # y (bytes 0x20000..) overlaps the last 48 mask bytes
])
def test_forward_bool_rejects_bad_arguments(kw):
    assert _fwd_bool(**kw) == INVALID
    assert binding.sms_last_error().startswith("sms_forward_bool")


def test_forward_bool_mask_extent_is_counted_in_bytes():
    # a byte mask of 64 elements ends 64 bytes after its start: y may begin
    # right there even for fp32 x, where an additive mask would be 256 bytes
    if torch.cuda.is_available():
        pytest.skip("host-only check")
    assert _fwd_bool(mask=0x20000 - 64, dtype=0) == binding.SMS_ERR_CUDA
    assert _fwd(mask=0x20000 - 64, mask_numel=64, rows=8, cols=8) == INVALID


def test_forward_bool_paths():
    # the byte mask is read by every family (no forced path refuses it on the
    # host; without a device each reaches the device query); a no-op stays a no-op
    if torch.cuda.is_available():
        pytest.skip("host-only check")
    for path, want in [(sms.SMS_PATH_RING, binding.SMS_ERR_CUDA), (sms.SMS_PATH_CTA, binding.SMS_ERR_CUDA),
                       (sms.SMS_PATH_STREAM, binding.SMS_ERR_CUDA), (sms.SMS_PATH_WARP, binding.SMS_ERR_CUDA),
                       (sms.SMS_PATH_ONLINE, binding.SMS_ERR_CUDA), (sms.SMS_PATH_AUTO, binding.SMS_ERR_CUDA)]:
        prev = sms.sms_set_forced_path(path)
        try:
            assert _fwd_bool() == want, path
        finally:
            sms.sms_set_forced_path(prev)
    assert _fwd_bool(rows=0, mask=None, x=None, y=None) == binding.SMS_OK


def test_build_compiles_every_kernel_source():
    # a translation unit left out of the build list would drop its kernels
    # (and, for the boolean-mask warp kernels, an entry point's launches)
    from scaled_masked_softmax_gb300 import build

    cu = sorted(f for f in os.listdir(build.CSRC) if f.endswith(".cu"))
    assert sorted(build.SOURCES) == cu


def _attn(**kw):
    a = dict(q=0x100000, k=0x200000, v=0x300000, mask=None, mask_numel=0, sb=0, sh=0, mbool=0, o=0x400000,
             lse=0x500000, B=1, H=2, S=16, D=64, scale=0.125, causal=0, dtype=binding.SMS_BF16, stream=None)
    a.update(kw)
    return binding.lib().sms_attention_forward(a["q"], a["k"], a["v"], a["mask"], a["mask_numel"], a["sb"], a["sh"],
                                               a["mbool"], a["o"], a["lse"], a["B"], a["H"], a["S"], a["D"],
                                               a["scale"], a["causal"], a["dtype"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(dtype=binding.SMS_F32), UNSUPPORTED), (dict(D=96), UNSUPPORTED), (dict(D=256), UNSUPPORTED),
    (dict(dtype=7), INVALID), (dict(q=None), INVALID), (dict(v=None), INVALID), (dict(o=None), INVALID),
    (dict(k=0x200008), INVALID), (dict(o=0x400004), INVALID), (dict(lse=0x500002), INVALID),
    (dict(B=-1), INVALID), (dict(scale=float("nan")), INVALID),
    (dict(o=0x100000), INVALID),  # o aliases q
    (dict(lse=0x400010), INVALID),  # lse inside o
    (dict(mask=0x600000, mask_numel=16 * 16 - 1), INVALID),  # [S,S] mask one element short
    (dict(mask=0x600000, mask_numel=512, sb=-1), INVALID), (dict(mask=0x600008, mask_numel=512), INVALID),
    (dict(mask=0x600000, mask_numel=256, sh=256), INVALID),  # [1,H,S,S] needs 512
])
def test_attention_rejects_bad_arguments(kw, status):
    assert _attn(**kw) == status
    assert binding.lib().sms_last_error().decode().startswith("sms_attention_forward")


def test_attention_empty_problem_is_a_no_op():
    for kw in (dict(B=0), dict(H=0), dict(S=0)):
        assert _attn(q=None, k=None, v=None, o=None, **kw) in (INVALID, binding.SMS_OK)
    assert _attn(B=0) == binding.SMS_OK


def _attn_bwd(**kw):
    a = dict(q=0x100000, k=0x200000, v=0x300000, o=0x400000, do=0x500000, lse=0x600000, mask=None, mask_numel=0,
             sb=0, sh=0, mbool=0, dq=0x700000, dk=0x800000, dv=0x900000, ws=0xA00000, wsb=1 << 20, B=1, H=2, S=16,
             D=64, scale=0.125, causal=0, dtype=binding.SMS_BF16, stream=None)
    a.update(kw)
    return binding.lib().sms_attention_backward(a["q"], a["k"], a["v"], a["o"], a["do"], a["lse"], a["mask"],
                                                a["mask_numel"], a["sb"], a["sh"], a["mbool"], a["dq"], a["dk"],
                                                a["dv"], a["ws"], a["wsb"], a["B"], a["H"], a["S"], a["D"],
                                                a["scale"], a["causal"], a["dtype"], a["stream"])


def test_attention_backward_workspace_size():
    # the fp32 dQ accumulator in whole blocks of 128 queries, then one fp32 per query row
    assert binding.lib().sms_attention_backward_workspace(2, 3, 5, 64) == 2 * 3 * 128 * 64 * 4 + 2 * 3 * 5 * 4
    assert binding.lib().sms_attention_backward_workspace(1, 2, 300, 128) == 2 * 384 * 128 * 4 + 2 * 300 * 4
    assert binding.lib().sms_attention_backward_workspace(-1, 3, 5, 64) == -1


@pytest.mark.parametrize("kw,status", [
    (dict(dtype=binding.SMS_F32), UNSUPPORTED), (dict(D=32), UNSUPPORTED), (dict(lse=None), INVALID),
    (dict(do=None), INVALID), (dict(dk=None), INVALID), (dict(ws=None), INVALID),
    (dict(wsb=2 * 16 * 64 * 4), INVALID),  # one query row's delta short
    (dict(ws=0xA00008), INVALID), (dict(dq=0x100000), INVALID), (dict(dv=0x800000), INVALID),
    (dict(ws=0x700000), INVALID),  # workspace on top of dq
    (dict(lse=0x600002), INVALID), (dict(mask=0xB00000, mask_numel=255), INVALID),
])
def test_attention_backward_rejects_bad_arguments(kw, status):
    assert _attn_bwd(**kw) == status
    assert binding.lib().sms_last_error().decode().startswith("sms_attention_backward")


def test_test_stall_control_range():
    L = binding.lib()
    assert L.sms_set_test_stall(-1) == -1
    assert L.sms_set_test_stall(2_000_000_000) == -1
    prev = L.sms_set_test_stall(5000)
    assert L.sms_set_test_stall(prev) == 5000
