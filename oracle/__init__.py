"""fp64 CPU oracle for the fused ScaledMaskSoftmax (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline / reference arm may import this package.  The product path (the CUDA
library and its Python binding) never imports it, and this package imports
nothing from the product.

The arithmetic lives in ``oracle.c`` (plain C99, binary64); this module only
compiles it with gcc, loads it with ctypes and marshals arrays.  The forward is
the definition on the page "用CUDA自定义融合Softmax算子并封装进PyTorch" (§1.2 formula,
§2.1 max-subtracted form, §2.2 additive mask + causal flag, §3.1 causal
placement after the mask add); the backward is that page's §3.3 Jacobian
formula ``dx = (dy - sum(dy*y)) * y * scale``.  A fully masked row comes out
all zero (the "uniform or all zero, never divide" advice of the second
article's §4.2 table, read as all zero).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F32, F16, BF16, F64 = 0, 1, 2, 3

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, OpenMP if available)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + ".tmp"
    base = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]
    try:
        subprocess.run(base + ["-fopenmp", "-o", tmp, _SRC, "-lm"], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + ["-o", tmp, _SRC, "-lm"], check=True, capture_output=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            i64, dbl, vp, i32 = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
            lib.oracle_forward.argtypes = [vp, i64, vp, i64, vp, i64, i64, i64, vp, i32, dbl, i32, i32, vp]
            lib.oracle_forward.restype = i32
            lib.oracle_backward.argtypes = [vp, i32, vp, i32, i64, i64, dbl, vp]
            lib.oracle_backward.restype = i32
            lib.oracle_decode.argtypes = [vp, i64, i32]
            lib.oracle_decode.restype = dbl
            lib.oracle_decode_array.argtypes = [vp, i64, i32, vp]
            lib.oracle_decode_array.restype = i32
            lib.oracle_num_threads.restype = i32
            lib.oracle_set_num_threads.argtypes = [i32]
            _lib = lib
    return _lib


def _raw(a, dtype_code=None):
    """Return (contiguous numpy array holding the exact bytes, dtype code).

    Accepts numpy arrays (float32/float16/float64, or uint16 holding bf16 bits
    when dtype_code=BF16) and CPU torch tensors of float32/float16/bfloat16/float64.
    """
    try:
        import torch  # local import: the oracle itself does not need torch

        if isinstance(a, torch.Tensor):
            t = a.detach().to("cpu").contiguous()
            code = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16, torch.float64: F64}[t.dtype]
            if code in (F16, BF16):
                arr = t.view(torch.int16).numpy().view(np.uint16)
            else:
                arr = t.numpy()
            return np.ascontiguousarray(arr), code
    except ImportError:  # pragma: no cover
        pass
    arr = np.ascontiguousarray(a)
    if dtype_code is not None:
        return arr, dtype_code
    code = {np.dtype(np.float32): F32, np.dtype(np.float16): F16, np.dtype(np.float64): F64}[arr.dtype]
    return arr, code


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def decode(a, dtype_code=None) -> np.ndarray:
    """Widen every element to fp64 with the oracle's own decoders."""
    arr, code = _raw(a, dtype_code)
    flat = np.ascontiguousarray(arr.reshape(-1))
    out = np.empty(flat.size, dtype=np.float64)
    if _load().oracle_decode_array(flat.ctypes.data, flat.size, code, out.ctypes.data) != 0:
        raise ValueError("oracle_decode_array rejected its arguments")
    return out.reshape(arr.shape)


def decode_one(a, i: int, dtype_code=None) -> float:
    """Element i of the flattened array widened to fp64 (one decoder call)."""
    arr, code = _raw(a, dtype_code)
    flat = np.ascontiguousarray(arr.reshape(-1))
    return float(_load().oracle_decode(flat.ctypes.data, int(i), code))


def forward(x_rows, cols: int, scale: float, is_causal: bool = False, mask=None,
            mask_stride_b: int = 0, mask_stride_h: int = 0, heads: int = 1,
            row_index=None, dtype_code=None, key_lengths=None) -> np.ndarray:
    """fp64 forward of the rows in ``x_rows`` (any shape with last dim ``cols``).

    ``row_index`` gives each row's logical index in the [rows, cols] view (for
    the causal position q = r mod cols and the mask row); default 0..n-1.
    ``key_lengths`` (one integer per batch b = r // (heads*cols)) keeps only
    the keys j < key_lengths[b] (clamped to [0, cols]) of each row.  A mask of
    torch.bool / numpy bool or uint8 is a boolean mask: nonzero masks the key.
    ``scale`` is used as given (pass the float32 value the kernel sees).
    Returns an fp64 array shaped like x_rows.
    """
    xa, code = _raw(x_rows, dtype_code)
    if xa.size % cols:
        raise ValueError("x size is not a multiple of cols")
    n = xa.size // cols
    ma = None
    mask_kind = 0
    if mask is not None:
        try:
            import torch

            if isinstance(mask, torch.Tensor) and mask.dtype in (torch.bool, torch.uint8):
                mask = mask.detach().to("cpu").numpy()
        except ImportError:  # pragma: no cover
            pass
        if isinstance(mask, np.ndarray) and mask.dtype in (np.bool_, np.uint8):
            ma = np.ascontiguousarray(mask.astype(np.uint8))
            mask_kind = 1
        else:
            ma, mcode = _raw(mask, code)
            if mcode != code:
                raise ValueError("mask dtype must equal x dtype")
    ri = None
    if row_index is not None:
        ri = np.ascontiguousarray(np.asarray(row_index, dtype=np.int64).reshape(-1))
        if ri.size != n:
            raise ValueError("row_index length must equal the number of rows")
    la = None
    if key_lengths is not None:
        try:
            import torch

            if isinstance(key_lengths, torch.Tensor):
                key_lengths = key_lengths.detach().to("cpu").numpy()
        except ImportError:  # pragma: no cover
            pass
        la = np.ascontiguousarray(np.asarray(key_lengths, dtype=np.int64).clip(-(2 ** 31), 2 ** 31 - 1)
                                  .astype(np.int32).reshape(-1))
        last = (int(ri.max()) if ri is not None and ri.size else n - 1) // (cols * heads)
        if la.size <= last:
            raise ValueError("key_lengths has fewer entries than the rows' batches")
    y = np.empty((n, cols), dtype=np.float64)
    rc = _load().oracle_forward(
        xa.ctypes.data, n, None if ri is None else ri.ctypes.data, cols,
        None if ma is None else ma.ctypes.data, mask_stride_b, mask_stride_h, heads,
        None if la is None else la.ctypes.data, mask_kind, float(scale), int(bool(is_causal)), code, y.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_forward rejected its arguments")
    return y.reshape(xa.shape)


def backward(y_rows, dy_rows, cols: int, scale: float, y_dtype_code=None, dy_dtype_code=None) -> np.ndarray:
    """fp64 backward: dx = (dy - sum(dy*y)) * y * scale, row by row."""
    ya, ycode = _raw(y_rows, y_dtype_code)
    da, dcode = _raw(dy_rows, dy_dtype_code)
    if ya.size != da.size or ya.size % cols:
        raise ValueError("y and dy must have the same size, a multiple of cols")
    n = ya.size // cols
    dx = np.empty((n, cols), dtype=np.float64)
    rc = _load().oracle_backward(ya.ctypes.data, ycode, da.ctypes.data, dcode, n, cols, float(scale), dx.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_backward rejected its arguments")
    return dx.reshape(ya.shape)

