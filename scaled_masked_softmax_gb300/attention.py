"""PyTorch-facing fused attention: O = softmax(Q K^T * scale + mask, causal) V.

The next step after the fused softmax on the source pages: the second article
(pnsm.cn/news/1983787) §4.4 and "从GEMM到Transformer：手写CUDA算子优化的完整路线与性能调优实践"
§2.2 fuse the score product, the scaled and masked softmax and the product with
V into one kernel that never stores the [S, S] scores.  Here that kernel runs
on the tensor cores (libsms: sms_attention_forward / sms_attention_backward);
PyTorch only provides memory and the current stream.

q, k, v are [B, H, S, D] fp16 or bf16 tensors (D = 64 or 128).  The mask takes
the shapes of the fused softmax (``functional.mask_layout``): [S, S],
[B, 1, S, S] or [B, H, S, S], additive of q's dtype, or torch.bool / uint8
with true = masked key.
"""
from __future__ import annotations

import math
from typing import Optional

import torch

from . import binding
from .functional import _aligned, mask_layout

_DT = {torch.float16: binding.SMS_F16, torch.bfloat16: binding.SMS_BF16}


def _mask_args(mask, q):
    if mask is None:
        return None, 0, 0, 0, False, None
    if mask.device != q.device:
        raise ValueError("mask must be on q's device")
    is_bool = mask.dtype in (torch.bool, torch.uint8)
    if not is_bool and mask.dtype != q.dtype:
        raise ValueError("an additive mask must have q's dtype")
    B, H, S, _ = q.shape
    sb, sh, _ = mask_layout((B, H, S, S), tuple(mask.shape))
    m = _aligned(mask.view(torch.uint8) if mask.dtype == torch.bool else mask)
    return m.data_ptr(), m.numel(), sb, sh, is_bool, m


def _check_qkv(q, k, v):
    if q.dim() != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k and v must all be [B, H, S, D] of one shape")
    if q.dtype not in _DT or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k and v must share one dtype, float16 or bfloat16")
    if not (q.is_cuda and k.device == q.device and v.device == q.device):
        raise ValueError("q, k and v must be CUDA tensors on one device")


def attention_forward(q, k, v, mask: Optional[torch.Tensor] = None, scale: Optional[float] = None,
                      is_causal: bool = False, return_lse: bool = False):
    """O (and, with ``return_lse``, the fp32 [B, H, S] log of each row's softmax
    denominator) of the fused attention."""
    _check_qkv(q, k, v)
    B, H, S, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    q, k, v = _aligned(q), _aligned(k), _aligned(v)
    mptr, mnum, sb, sh, is_bool, keep = _mask_args(mask, q)
    o = torch.empty_like(q)
    lse = torch.empty(B, H, S, dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        st = torch.cuda.current_stream(q.device).cuda_stream
        binding.sms_attention_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), mptr, mnum, sb, sh, is_bool,
                                      o.data_ptr(), lse.data_ptr(), B, H, S, D, float(scale), is_causal, _DT[q.dtype],
                                      st)
    del keep
    return (o, lse) if return_lse else o


def attention_backward(q, k, v, o, lse, d_o, mask: Optional[torch.Tensor] = None, scale: Optional[float] = None,
                       is_causal: bool = False):
    """(dQ, dK, dV) of sum(dO * O) for the forward that produced o and lse
    (the same q, k, v, mask, scale and causal flag).  The fp32 scratch the
    kernels need is taken from PyTorch's allocator for the call."""
    _check_qkv(q, k, v)
    B, H, S, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    q, k, v, o, d_o = _aligned(q), _aligned(k), _aligned(v), _aligned(o), _aligned(d_o)
    if o.shape != q.shape or d_o.shape != q.shape or o.dtype != q.dtype or d_o.dtype != q.dtype:
        raise ValueError("o and d_o must match q in shape and dtype")
    lse = _aligned(lse.to(torch.float32))
    mptr, mnum, sb, sh, is_bool, keep = _mask_args(mask, q)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    nws = binding.sms_attention_backward_workspace(B, H, S, D)
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=q.device)
    with torch.cuda.device(q.device):
        st = torch.cuda.current_stream(q.device).cuda_stream
        binding.sms_attention_backward(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), d_o.data_ptr(),
                                       lse.data_ptr(), mptr, mnum, sb, sh, is_bool, dq.data_ptr(), dk.data_ptr(),
                                       dv.data_ptr(), ws.data_ptr(), ws.numel(), B, H, S, D, float(scale), is_causal,
                                       _DT[q.dtype], st)
    del keep, ws
    return dq, dk, dv


class FusedAttentionFunction(torch.autograd.Function):
    """O = fused attention of (q, k, v); the backward reruns the tensor-core
    backward from q, k, v, O and the saved per-row log-sum-exp.  No gradient
    flows to the mask, the scale or the causal flag."""

    @staticmethod
    def forward(ctx, q, k, v, mask, scale, is_causal):
        o, lse = attention_forward(q, k, v, mask, scale, is_causal, return_lse=True)
        ctx.save_for_backward(q, k, v, o, lse, mask if mask is not None else torch.empty(0, device=q.device))
        ctx.has_mask = mask is not None
        ctx.scale, ctx.is_causal = scale, is_causal
        return o

    @staticmethod
    def backward(ctx, d_o):
        q, k, v, o, lse, mask = ctx.saved_tensors
        dq, dk, dv = attention_backward(q, k, v, o, lse, d_o.contiguous(), mask if ctx.has_mask else None, ctx.scale,
                                        ctx.is_causal)
        return dq, dk, dv, None, None, None


def fused_attention(q, k, v, mask: Optional[torch.Tensor] = None, scale: Optional[float] = None,
                    is_causal: bool = False):
    """Differentiable O = softmax(Q K^T * scale + mask, causal) V on the tensor cores."""
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    return FusedAttentionFunction.apply(q, k, v, mask, float(scale), bool(is_causal))
