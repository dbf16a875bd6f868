"""Shared helpers for the GPU parity tests: run the CUDA path, run the oracle
on the same bytes, and compare within the stated tolerances."""
from __future__ import annotations

import contextlib

import numpy as np
import torch

import oracle
import scaled_masked_softmax_gb300 as sms
from scaled_masked_softmax_gb300 import workloads

# |y - y_ref| bounds per output dtype (fp32 2e-6, fp16 1e-3, bf16 8e-3 absolute)
FWD_ATOL = {torch.float32: 2e-6, torch.float16: 1e-3, torch.bfloat16: 8e-3}
# unit roundoff of the stored dtype, used by the backward bound
UNIT = {torch.float32: 2.0 ** -24, torch.float16: 2.0 ** -11, torch.bfloat16: 2.0 ** -8}

PATHS = {"auto": sms.SMS_PATH_AUTO, "warp": sms.SMS_PATH_WARP, "cta": sms.SMS_PATH_CTA, "online": sms.SMS_PATH_ONLINE,
         "stream": sms.SMS_PATH_STREAM, "ring": sms.SMS_PATH_RING}


@contextlib.contextmanager
def grid_limit(ctas: int):
    prev = sms.sms_set_grid_limit(ctas)
    try:
        yield
    finally:
        sms.sms_set_grid_limit(prev)


@contextlib.contextmanager
def forced_path(name: str):
    prev = sms.sms_set_forced_path(PATHS[name])
    try:
        yield
    finally:
        sms.sms_set_forced_path(prev)


def to_np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def oracle_forward(inp, w, row_idx=None):
    """fp64 oracle of the rows ``row_idx`` (all rows if None) of workload inputs."""
    x = inp["x"]
    if row_idx is None:
        xr = x.cpu()
        ri = None
    else:
        ri = np.asarray(row_idx, dtype=np.int64)
        xr = x[torch.as_tensor(ri, device=x.device)].cpu()
    mask = inp["mask"].cpu() if inp["mask"] is not None else None
    return oracle.forward(xr, w.cols, w.scale, w.is_causal, mask, inp["mask_stride_b"], inp["mask_stride_h"],
                          inp["heads"], row_index=ri)


def gpu_forward(inp, w):
    x = inp["x"]
    return sms.forward(x.view(*shape_of(w)) if w.rows == w.B * w.H * w.S else x, inp["mask"], w.scale,
                       w.is_causal).reshape(w.rows, w.cols)


def shape_of(w):
    return (w.B, w.H, w.S, w.S)


def raw_forward(inp, w, y=None):
    """Forward through the C ABI with explicit strides (any rows, any mask layout)."""
    x = inp["x"]
    y = torch.empty_like(x) if y is None else y
    m = inp["mask"]
    dt = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}[x.dtype]
    sms.sms_forward(x.data_ptr(), None if m is None else m.data_ptr(), 0 if m is None else m.numel(),
                    inp["mask_stride_b"], inp["mask_stride_h"], inp["heads"], y.data_ptr(), w.rows, w.cols,
                    w.scale, w.is_causal, dt, torch.cuda.current_stream().cuda_stream)
    return y


def raw_forward_lengths(x, lengths, heads, w, y=None):
    """sms_forward_lengths through the C ABI (rows of x, per-batch key lengths)."""
    y = torch.empty_like(x) if y is None else y
    dt = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}[x.dtype]
    sms.sms_forward_lengths(x.data_ptr(), lengths.data_ptr(), heads, y.data_ptr(), w.rows, w.cols, w.scale,
                            w.is_causal, dt, torch.cuda.current_stream().cuda_stream)
    return y


def raw_backward_lengths(y, dy, lengths, heads, w, causal_hint, dx=None):
    dx = torch.empty_like(y) if dx is None else dx
    dt = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}[y.dtype]
    sms.sms_backward_lengths(y.data_ptr(), dy.data_ptr(), dx.data_ptr(), lengths.data_ptr(), heads, w.rows, w.cols,
                             w.scale, causal_hint, dt, torch.cuda.current_stream().cuda_stream)
    return dx


def raw_backward(y, dy, w, causal_hint, dx=None):
    dx = torch.empty_like(y) if dx is None else dx
    dt = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}[y.dtype]
    sms.sms_backward(y.data_ptr(), dy.data_ptr(), dx.data_ptr(), w.rows, w.cols, w.scale, causal_hint, dt,
                     torch.cuda.current_stream().cuda_stream)
    return dx


def check_forward(y_gpu: np.ndarray, y_ref: np.ndarray, dtype, what=""):
    atol = FWD_ATOL[dtype]
    err = np.abs(y_gpu - y_ref)
    worst = float(err.max()) if err.size else 0.0
    assert worst <= atol, f"{what}: max |y - y_ref| = {worst:.3e} > {atol:.1e}"
    # every position the fp64 definition makes exactly 0 (masked, causal, or
    # underflowed) is exactly 0
    zero = y_ref == 0.0
    assert np.all(y_gpu[zero] == 0.0), f"{what}: {int(np.sum(y_gpu[zero] != 0))} positions should be exactly 0"
    assert np.all(np.isfinite(y_gpu)), f"{what}: non-finite output"
    if dtype == torch.float32 and y_ref.size:
        rs = y_ref.sum(-1)
        live = rs > 0.5  # rows that are not fully masked
        dev = np.abs(1.0 - y_gpu.sum(-1)[live])
        assert dev.size == 0 or float(dev.max()) <= 1e-5, f"{what}: |1 - sum y| = {float(dev.max()):.2e}"
    return worst


def check_backward(dx_gpu: np.ndarray, y: np.ndarray, dy: np.ndarray, scale: float, dtype, what=""):
    """dx against the oracle on the same stored y and dy.

    fp32: max|dx - ref| / max|ref| <= 1e-5 per tensor.  fp16/bf16 (no bound is
    stated on the pages): |dx - ref| <= 2u (|ref| + |scale| |y| (|dy| + |dot|)) + 1e-7
    elementwise, u the unit roundoff of the dtype.
    """
    ref = oracle.backward(y, dy, y.shape[-1], scale)
    if dtype == torch.float32:
        denom = max(float(np.abs(ref).max()), 1e-30)
        rel = float(np.abs(dx_gpu - ref).max()) / denom
        assert rel <= 1e-5, f"{what}: relative error {rel:.3e} > 1e-5"
        return rel
    y64 = y if isinstance(y, np.ndarray) else to_np64(y)
    dy64 = dy if isinstance(dy, np.ndarray) else to_np64(dy)
    dot = np.sum(y64 * dy64, axis=-1, keepdims=True)
    bound = 2 * UNIT[dtype] * (np.abs(ref) + abs(scale) * np.abs(y64) * (np.abs(dy64) + np.abs(dot))) + 1e-7
    excess = np.abs(dx_gpu - ref) - bound
    assert float(excess.max()) <= 0, f"{what}: backward error exceeds bound by {float(excess.max()):.3e}"
    return float(np.abs(dx_gpu - ref).max())


def make(w, device="cuda"):
    return workloads.make_inputs(w, device=device)


def raw_forward_bool(x, mask, sb, sh, heads, w, y=None):
    """sms_forward_bool through the C ABI: ``mask`` is a bool / uint8 device
    tensor read one byte per element (nonzero = masked)."""
    y = torch.empty_like(x) if y is None else y
    dt = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}[x.dtype]
    sms.sms_forward_bool(x.data_ptr(), mask.data_ptr(), mask.numel(), sb, sh, heads, y.data_ptr(), w.rows, w.cols,
                         w.scale, w.is_causal, dt, torch.cuda.current_stream().cuda_stream)
    return y


# ------------------------------------------------------- whole-tensor parity ---
# The full-size workloads are checked on every row: the fp64 oracle runs on the
# host over chunks of rows (OpenMP over rows), its result is copied to the
# device, and the comparison (the same bounds as check_forward /
# check_backward) runs there in fp64.

def _chunk_rows(w, elems=1 << 25):
    step = max(1, elems // w.cols)
    return [(r0, min(w.rows, r0 + step)) for r0 in range(0, w.rows, step)]


class FullCheck:
    """Accumulates the whole-tensor bounds over row chunks."""

    def __init__(self, dtype, what):
        self.dtype, self.what = dtype, what
        self.fwd_worst = 0.0
        self.bwd_err = 0.0   # max |dx - ref| (fp32: over the tensor)
        self.bwd_ref = 0.0   # max |ref| (fp32 per-tensor relative bound)
        self.rows = 0

    def forward(self, y_dev: torch.Tensor, ref_np: np.ndarray, r0: int):
        ref = torch.from_numpy(ref_np).to(y_dev.device)
        y = y_dev.to(torch.float64)
        assert bool(torch.isfinite(y).all()), f"{self.what}: non-finite output near row {r0}"
        err = (y - ref).abs()
        worst = float(err.max()) if err.numel() else 0.0
        self.fwd_worst = max(self.fwd_worst, worst)
        assert worst <= FWD_ATOL[self.dtype], \
            f"{self.what}: max |y - y_ref| = {worst:.3e} > {FWD_ATOL[self.dtype]:.1e} in rows from {r0}"
        bad = int(((ref == 0) & (y != 0)).sum())
        assert bad == 0, f"{self.what}: {bad} positions should be exactly 0 in rows from {r0}"
        if self.dtype == torch.float32:
            live = ref.sum(-1) > 0.5
            dev = (1.0 - y.sum(-1))[live].abs()
            assert dev.numel() == 0 or float(dev.max()) <= 1e-5, \
                f"{self.what}: |1 - sum y| = {float(dev.max()):.2e} in rows from {r0}"
        self.rows += y_dev.shape[0]

    def backward(self, dx_dev: torch.Tensor, y_dev: torch.Tensor, dy_dev: torch.Tensor, ref_np: np.ndarray,
                 scale: float, r0: int):
        ref = torch.from_numpy(ref_np).to(dx_dev.device)
        dx = dx_dev.to(torch.float64)
        assert bool(torch.isfinite(dx).all()), f"{self.what}: non-finite gradient near row {r0}"
        err = (dx - ref).abs()
        if self.dtype == torch.float32:
            self.bwd_err = max(self.bwd_err, float(err.max()))
            self.bwd_ref = max(self.bwd_ref, float(ref.abs().max()))
            return
        y = y_dev.to(torch.float64)
        dy = dy_dev.to(torch.float64)
        dot = (y * dy).sum(-1, keepdim=True)
        bound = 2 * UNIT[self.dtype] * (ref.abs() + abs(scale) * y.abs() * (dy.abs() + dot.abs())) + 1e-7
        excess = float((err - bound).max())
        assert excess <= 0, f"{self.what}: backward error exceeds bound by {excess:.3e} in rows from {r0}"
        self.bwd_err = max(self.bwd_err, float(err.max()))

    def finish_backward(self):
        if self.dtype == torch.float32:
            rel = self.bwd_err / max(self.bwd_ref, 1e-30)
            assert rel <= 1e-5, f"{self.what}: backward relative error {rel:.3e} > 1e-5"


def check_all_rows(w, inp, y, dx=None, what="", key_lengths=None, bool_mask=None):
    """Every row of y (and dx, the backward of y against inp['dy']) against the
    oracle.  key_lengths: the per-batch lengths the forward used instead of
    the mask; bool_mask: the byte mask it used instead of the additive one."""
    chk = FullCheck(w.torch_dtype, what)
    mask = None
    if key_lengths is None:
        mask = bool_mask if bool_mask is not None else inp["mask"]
        mask = mask.cpu() if mask is not None else None
    L = key_lengths.cpu() if key_lengths is not None else None
    for r0, r1 in _chunk_rows(w):
        xr = inp["x"][r0:r1].cpu()
        ri = np.arange(r0, r1, dtype=np.int64)
        if L is not None:
            ref = oracle.forward(xr, w.cols, w.scale, w.is_causal, heads=w.H, key_lengths=L, row_index=ri)
        else:
            ref = oracle.forward(xr, w.cols, w.scale, w.is_causal, mask, inp["mask_stride_b"], inp["mask_stride_h"],
                                 inp["heads"], row_index=ri)
        chk.forward(y[r0:r1], ref, r0)
        if dx is not None:
            yr, dyr = y[r0:r1], inp["dy"][r0:r1]
            dref = oracle.backward(yr.cpu(), dyr.cpu(), w.cols, w.scale)
            chk.backward(dx[r0:r1], yr, dyr, dref, w.scale, r0)
    if dx is not None:
        chk.finish_backward()
    assert chk.rows == w.rows
    return chk
