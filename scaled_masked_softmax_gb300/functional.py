"""PyTorch-facing API of the fused ScaledMaskSoftmax (autograd included).

The shape conventions follow the page "用CUDA自定义融合Softmax算子并封装进PyTorch":
x is an attention-score tensor [B, H, S, S] (any leading dims; rows = numel /
size(-1), §4.2), the mask is additive, of x's dtype, and may be omitted (§2.2);
``ScaledMaskSoftmaxFunction`` keeps only the output y for the backward and
returns no gradient for mask, scale or is_causal (§4.3).  A torch.bool (or
uint8) mask is a boolean mask, true = masked key: §2.2 converts it to the
additive ``mask * -inf`` before the kernel (and §5.1 warns that adding it as
1.0 is wrong); here the kernel reads the bytes itself, with the result of
that additive mask bit for bit and a quarter / half of its bytes.  A key-padding
mask can instead be given as ``key_lengths`` (int32 [B], the valid keys of
each batch): the same result as the additive mask with -inf beyond L_b, with
no mask tensor read and the padded scores never read.

PyTorch provides only memory, device placement and the current stream here;
the computation runs in libsms through the C ABI.
"""
from __future__ import annotations

import math
from typing import Optional

import torch

from . import binding

_DTYPE_CODE = {torch.float32: binding.SMS_F32, torch.float16: binding.SMS_F16, torch.bfloat16: binding.SMS_BF16}


def _aligned(t: torch.Tensor) -> torch.Tensor:
    """Contiguous, 16-byte aligned storage (clones a misaligned view)."""
    t = t.contiguous()
    if t.numel() and t.data_ptr() % 16:
        t = t.clone()
    return t


def mask_layout(x_shape, mask_shape):
    """(mask_stride_b, mask_stride_h, heads) for a mask broadcast against x.

    x is read as [B, H, S, S] (H = size(-3), B = the product of the leading
    dims).  Supported masks, right-aligned against x: [S,S]; [.., 1, S, S]
    (broadcast over heads) or [.., H, S, S]; leading dims all 1 (shared by
    every batch) or all equal to x's.
    """
    S = x_shape[-1]
    nd = len(x_shape)
    md = len(mask_shape)
    if md < 2 or md > nd or tuple(mask_shape[-2:]) != (x_shape[-2], S):
        raise ValueError(f"mask shape {tuple(mask_shape)} does not broadcast to x shape {tuple(x_shape)} "
                         "over the last two dims")
    H = x_shape[-3] if nd >= 3 else 1
    if md == 2:
        return 0, 0, H
    Hm = mask_shape[-3]
    if Hm not in (1, H):
        raise ValueError(f"mask head dim {Hm} must be 1 or {H}")
    lead_x = list(x_shape[:-3])
    lead_m = [1] * (len(lead_x) - (md - 3)) + list(mask_shape[:-3])
    if all(d == 1 for d in lead_m):
        full_b = False
    elif lead_m == lead_x:
        full_b = True
    else:
        raise ValueError(f"mask leading dims {tuple(mask_shape[:-3])} must be all 1 or equal x's {tuple(lead_x)}")
    sh = S * S if (Hm == H and H > 1) else 0
    sb = (Hm * S * S) if full_b else 0
    return sb, sh, H


def _key_lengths(key_lengths: torch.Tensor, x_shape, device) -> tuple:
    """(contiguous int32 lengths, heads) for x read as [B, H, S, S]."""
    if len(x_shape) < 2 or x_shape[-2] != x_shape[-1]:
        raise ValueError("key_lengths needs square score matrices (x.shape[-2] == x.shape[-1])")
    if key_lengths.dtype != torch.int32 or key_lengths.device != device:
        raise TypeError("key_lengths must be an int32 tensor on x's device")
    H = x_shape[-3] if len(x_shape) >= 3 else 1
    B = math.prod(x_shape[:-3]) if len(x_shape) > 3 else 1
    if key_lengths.numel() != B:
        raise ValueError(f"key_lengths has {key_lengths.numel()} entries, x has {B} batches")
    return key_lengths.contiguous(), H


def forward(x: torch.Tensor, mask: Optional[torch.Tensor] = None, scale: float = 1.0, is_causal: bool = False,
            out: Optional[torch.Tensor] = None, key_lengths: Optional[torch.Tensor] = None) -> torch.Tensor:
    """y = softmax(x * scale + mask) over the last dim, j > q masked if is_causal,
    keys j >= key_lengths[b] masked when key_lengths is given.  A torch.bool
    mask masks the keys where it is true (score -inf)."""
    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor (there is no CPU path)")
    if x.dtype not in _DTYPE_CODE:
        raise TypeError(f"x dtype {x.dtype} not supported (float32, float16, bfloat16)")
    if x.dim() < 1 or x.shape[-1] == 0:
        raise ValueError("x must have a non-empty last dim")
    cols = x.shape[-1]
    if (is_causal or mask is not None) and (x.dim() < 2 or x.shape[-2] != cols):
        raise ValueError("a mask or is_causal needs square score matrices (x.shape[-2] == x.shape[-1])")
    x = _aligned(x)
    rows = x.numel() // cols
    dt = _DTYPE_CODE[x.dtype]
    y = torch.empty_like(x) if out is None else out
    if y.shape != x.shape or y.dtype != x.dtype or y.device != x.device or not y.is_contiguous() or \
            (y.numel() and y.data_ptr() % 16):
        raise ValueError("out must be a contiguous, 16-byte aligned tensor like x")
    mptr, mnum, sb, sh, heads = None, 0, 0, 0, (x.shape[-3] if x.dim() >= 3 else 1)
    mask_bool = False
    if key_lengths is not None:
        if mask is not None:
            raise ValueError("give either an additive mask or key_lengths, not both")
        lengths, heads = _key_lengths(key_lengths, x.shape, x.device)
        if rows == 0:
            return y
        with torch.cuda.device(x.device):
            stream = torch.cuda.current_stream(x.device).cuda_stream
            binding.sms_forward_lengths(x.data_ptr(), lengths.data_ptr(), heads, y.data_ptr(), rows, cols,
                                        float(scale), bool(is_causal), dt, stream)
        return y
    if mask is not None:
        mask_bool = mask.dtype in (torch.bool, torch.uint8)
        if not mask_bool and mask.dtype != x.dtype:
            raise TypeError(f"mask dtype {mask.dtype} must equal x dtype {x.dtype}, or be torch.bool")
        if mask.device != x.device:
            raise ValueError("mask must be on x's device")
        sb, sh, heads = mask_layout(x.shape, mask.shape)
        mask = _aligned(mask)
        mptr, mnum = mask.data_ptr(), mask.numel()
    if rows == 0:
        return y
    with torch.cuda.device(x.device):
        stream = torch.cuda.current_stream(x.device).cuda_stream
        if mask_bool:  # torch.bool stores one byte per element, 0 or 1
            binding.sms_forward_bool(x.data_ptr(), mptr, mnum, sb, sh, heads, y.data_ptr(), rows, cols, float(scale),
                                     bool(is_causal), dt, stream)
            return y
        binding.sms_forward(x.data_ptr(), mptr, mnum, sb, sh, heads, y.data_ptr(), rows, cols, float(scale),
                            bool(is_causal), dt, stream)
    return y


def backward(y: torch.Tensor, dy: torch.Tensor, scale: float = 1.0, is_causal_hint: bool = False,
             out: Optional[torch.Tensor] = None, key_lengths: Optional[torch.Tensor] = None) -> torch.Tensor:
    """dx = (dy - sum(dy*y)) * y * scale over the last dim; key_lengths (and
    is_causal_hint) promise y == 0 beyond them, so those positions are not read."""
    if not (y.is_cuda and dy.is_cuda):
        raise ValueError("y and dy must be CUDA tensors (there is no CPU path)")
    if y.dtype not in _DTYPE_CODE or dy.dtype != y.dtype:
        raise TypeError("y and dy must share a dtype among float32, float16, bfloat16")
    if y.shape != dy.shape:
        raise ValueError("y and dy must have the same shape")
    cols = y.shape[-1]
    if is_causal_hint and (y.dim() < 2 or y.shape[-2] != cols):
        raise ValueError("the causal hint needs square score matrices")
    y = _aligned(y)
    dy = _aligned(dy)
    rows = y.numel() // cols if cols else 0
    dx = torch.empty_like(y) if out is None else out
    if dx.shape != y.shape or dx.dtype != y.dtype or not dx.is_contiguous() or (dx.numel() and dx.data_ptr() % 16):
        raise ValueError("out must be a contiguous, 16-byte aligned tensor like y")
    if rows == 0:
        return dx
    if key_lengths is not None:
        lengths, heads = _key_lengths(key_lengths, y.shape, y.device)
        with torch.cuda.device(y.device):
            stream = torch.cuda.current_stream(y.device).cuda_stream
            binding.sms_backward_lengths(y.data_ptr(), dy.data_ptr(), dx.data_ptr(), lengths.data_ptr(), heads, rows,
                                         cols, float(scale), bool(is_causal_hint), _DTYPE_CODE[y.dtype], stream)
        return dx
    with torch.cuda.device(y.device):
        stream = torch.cuda.current_stream(y.device).cuda_stream
        binding.sms_backward(y.data_ptr(), dy.data_ptr(), dx.data_ptr(), rows, cols, float(scale),
                             bool(is_causal_hint), _DTYPE_CODE[y.dtype], stream)
    return dx


class ScaledMaskSoftmaxFunction(torch.autograd.Function):
    """Saves y (not x) for backward; no gradient for mask, scale, is_causal or
    key_lengths."""

    @staticmethod
    def forward(ctx, x, mask, scale, is_causal, key_lengths=None):
        y = forward(x, mask, scale, is_causal, key_lengths=key_lengths)
        ctx.save_for_backward(y)
        ctx.key_lengths = key_lengths
        ctx.scale = float(scale)
        ctx.is_causal = bool(is_causal)
        return y

    @staticmethod
    def backward(ctx, grad_y):
        (y,) = ctx.saved_tensors
        dx = backward(y, grad_y, ctx.scale, is_causal_hint=ctx.is_causal, key_lengths=ctx.key_lengths)
        return dx, None, None, None, None


def scaled_mask_softmax(x: torch.Tensor, mask: Optional[torch.Tensor] = None, scale: float = 1.0,
                        is_causal: bool = False, key_lengths: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Fused softmax(x * scale + mask) over the last dim, differentiable in x.
    key_lengths (int32 [B]) masks keys j >= key_lengths[b] without a mask tensor."""
    if not math.isfinite(float(scale)):
        raise ValueError("scale must be finite")
    return ScaledMaskSoftmaxFunction.apply(x, mask, scale, is_causal, key_lengths)
