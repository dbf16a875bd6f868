"""ctypes binding of libsms (include/sms.h): the same entry points, same names.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind these calls.  There is no CPU fallback - if libsms.so has not
been built, loading raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsms.so")

SMS_F32, SMS_F16, SMS_BF16 = 0, 1, 2
SMS_ATTN_STATIC_SCRATCH_BYTES = 32 << 20  # include/sms.h: the static scratch of sms_attention_backward_static
SMS_OK, SMS_ERR_INVALID_ARG, SMS_ERR_UNSUPPORTED, SMS_ERR_CUDA = 0, 1, 2, 3
SMS_PATH_AUTO, SMS_PATH_WARP, SMS_PATH_CTA, SMS_PATH_ONLINE, SMS_PATH_STREAM, SMS_PATH_RING = 0, 1, 2, 3, 4, 5
PATH_NAMES = {SMS_PATH_AUTO: "auto", SMS_PATH_WARP: "warp", SMS_PATH_CTA: "cta", SMS_PATH_ONLINE: "online",
              SMS_PATH_STREAM: "stream", SMS_PATH_RING: "ring"}

# every function include/sms.h declares: name -> (restype, argtypes)
_i64, _i32, _f32, _vp, _cp = ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_char_p
SIGNATURES = {
    "sms_forward": (_i32, [_vp, _vp, _i64, _i64, _i64, _i64, _vp, _i64, _i64, _f32, _i32, _i32, _vp]),
    "sms_forward_bool": (_i32, [_vp, _vp, _i64, _i64, _i64, _i64, _vp, _i64, _i64, _f32, _i32, _i32, _vp]),
    "sms_backward": (_i32, [_vp, _vp, _vp, _i64, _i64, _f32, _i32, _i32, _vp]),
    "sms_forward_lengths": (_i32, [_vp, _vp, _i64, _vp, _i64, _i64, _f32, _i32, _i32, _vp]),
    "sms_backward_lengths": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _f32, _i32, _i32, _vp]),
    "sms_attention_forward": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _vp, _vp, _i64, _i64, _i64, _i64,
                                     _f32, _i32, _i32, _vp]),
    "sms_attention_backward": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _vp, _vp, _vp, _vp,
                                      _i64, _i64, _i64, _i64, _i64, _f32, _i32, _i32, _vp]),
    "sms_attention_backward_workspace": (_i64, [_i64, _i64, _i64, _i64]),
    "sms_attention_backward_static": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _vp, _vp, _vp,
                                             _i64, _i64, _i64, _i64, _f32, _i32, _i32, _vp]),
    "sms_status_string": (_cp, [_i32]),
    "sms_last_error": (_cp, []),
    "sms_set_forced_path": (_i32, [_i32]),
    "sms_set_grid_limit": (_i32, [_i32]),
    "sms_select_path": (_i32, [_i64, _i64, _i32, _i32]),
    "sms_last_path": (_i32, []),
    "sms_launch_count": (_i64, []),
    "sms_set_test_stall": (_i64, [_i64]),
    "sms_device_error": (_i32, [_vp]),
    "sms_version": (_i32, []),
}

_lock = threading.Lock()
_lib = None


class SmsError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


def lib() -> ctypes.CDLL:
    """Load libsms.so (built in-tree by ``scaled_masked_softmax_gb300.build``)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"libsms.so is not built ({LIB_PATH} missing); run "
                        "`python -c 'import __graft_entry__ as g; g.build()'` first")
                h = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in SIGNATURES.items():
                    fn = getattr(h, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = h
    return _lib


def _check(status: int) -> None:
    if status != SMS_OK:
        L = lib()
        msg = L.sms_last_error().decode() or L.sms_status_string(status).decode()
        raise SmsError(status, msg)


def sms_forward(x, mask, mask_numel, mask_stride_b, mask_stride_h, heads, y, rows, cols, scale, is_causal, dtype,
                stream) -> None:
    """Raw pointers in, status checked: see include/sms.h."""
    _check(lib().sms_forward(x, mask, mask_numel, mask_stride_b, mask_stride_h, heads, y, rows, cols, scale,
                             int(bool(is_causal)), dtype, stream))


def sms_forward_bool(x, mask, mask_numel, mask_stride_b, mask_stride_h, heads, y, rows, cols, scale, is_causal,
                     dtype, stream) -> None:
    """Boolean mask (one byte per element, nonzero = masked): see include/sms.h."""
    _check(lib().sms_forward_bool(x, mask, mask_numel, mask_stride_b, mask_stride_h, heads, y, rows, cols, scale,
                                  int(bool(is_causal)), dtype, stream))


def sms_backward(y, dy, dx, rows, cols, scale, is_causal_hint, dtype, stream) -> None:
    _check(lib().sms_backward(y, dy, dx, rows, cols, scale, int(bool(is_causal_hint)), dtype, stream))


def sms_forward_lengths(x, lengths, heads, y, rows, cols, scale, is_causal, dtype, stream) -> None:
    _check(lib().sms_forward_lengths(x, lengths, heads, y, rows, cols, scale, int(bool(is_causal)), dtype, stream))


def sms_backward_lengths(y, dy, dx, lengths, heads, rows, cols, scale, is_causal_hint, dtype, stream) -> None:
    _check(lib().sms_backward_lengths(y, dy, dx, lengths, heads, rows, cols, scale, int(bool(is_causal_hint)), dtype,
                                      stream))


def sms_attention_forward(q, k, v, mask, mask_numel, mask_stride_b, mask_stride_h, mask_is_bool, o, lse, batch, heads,
                          seq, head_dim, scale, is_causal, dtype, stream) -> None:
    """Fused attention forward on the tensor cores: see include/sms.h."""
    _check(lib().sms_attention_forward(q, k, v, mask, mask_numel, mask_stride_b, mask_stride_h, int(bool(mask_is_bool)),
                                       o, lse, batch, heads, seq, head_dim, scale, int(bool(is_causal)), dtype,
                                       stream))


def sms_attention_backward(q, k, v, o, d_o, lse, mask, mask_numel, mask_stride_b, mask_stride_h, mask_is_bool, dq, dk,
                           dv, workspace, workspace_bytes, batch, heads, seq, head_dim, scale, is_causal, dtype,
                           stream) -> None:
    """Fused attention backward on the tensor cores: see include/sms.h."""
    _check(lib().sms_attention_backward(q, k, v, o, d_o, lse, mask, mask_numel, mask_stride_b, mask_stride_h,
                                        int(bool(mask_is_bool)), dq, dk, dv, workspace, workspace_bytes, batch, heads,
                                        seq, head_dim, scale, int(bool(is_causal)), dtype, stream))


def sms_attention_backward_workspace(batch, heads, seq, head_dim) -> int:
    return int(lib().sms_attention_backward_workspace(batch, heads, seq, head_dim))


def sms_set_forced_path(path: int) -> int:
    prev = lib().sms_set_forced_path(int(path))
    if prev < 0:
        raise ValueError(f"unknown path {path}")
    return prev


def sms_set_grid_limit(ctas: int) -> int:
    prev = lib().sms_set_grid_limit(int(ctas))
    if prev < 0:
        raise ValueError(f"bad CTA limit {ctas}")
    return prev


def sms_select_path(rows: int, cols: int, dtype: int, is_backward: bool = False) -> int:
    return lib().sms_select_path(rows, cols, dtype, int(bool(is_backward)))


def sms_last_path() -> int:
    return lib().sms_last_path()


def sms_launch_count() -> int:
    return lib().sms_launch_count()


def sms_set_test_stall(ns: int) -> int:
    prev = lib().sms_set_test_stall(int(ns))
    if prev < 0:
        raise ValueError(f"bad stall {ns}")
    return prev


def sms_device_error(stream) -> int:
    return lib().sms_device_error(stream)


def sms_version() -> int:
    return lib().sms_version()


def sms_status_string(status: int) -> str:
    return lib().sms_status_string(status).decode()


def sms_last_error() -> str:
    return lib().sms_last_error().decode()
