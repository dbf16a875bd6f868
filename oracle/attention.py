"""fp64 oracle of the fused attention step around the softmax (test infrastructure only).

The fusion the pages point to next: the second article (pnsm.cn/news/1983787)
§4.4 and the page "从GEMM到Transformer：手写CUDA算子优化的完整路线与性能调优实践"
§2.2 compute Q K^T -> scale and mask -> softmax -> multiply by V in one kernel,
without materialising the [B, H, S, S] score tensor.  This module is its plain
definition, in binary64:

    S_b,h = Q_b,h K_b,h^T            (matmul, a library primitive)
    P     = the softmax oracle of S with the same scale, mask and causal rule
            (oracle.forward: s = S*scale + mask, j > i masked under causal,
            fully masked rows all zero)
    O_b,h = P_b,h V_b,h              (matmul)

and its gradient, by the chain rule through the same three steps:

    dV = P^T dO,   dP = dO V^T,
    dS = oracle.backward(P, dP, scale)   (= scale * P * (dP - rowsum(P * dP)))
    dQ = dS K,     dK = dS^T Q.

Q, K, V and dO may be float32 / float16 / bfloat16 / float64 tensors or arrays;
every element is widened exactly to fp64 first (oracle.decode).  Only the test
suite and the benchmark's CPU legs may import this; the product never does.
"""
from __future__ import annotations

import numpy as np

from . import backward as _softmax_backward
from . import decode, forward as _softmax_forward


def _f64(a) -> np.ndarray:
    return np.asarray(decode(a), dtype=np.float64).reshape(tuple(a.shape))


def _bhsd(a, name):
    if a.ndim != 4:
        raise ValueError(f"{name} must be [B, H, S, D]")
    return a


def attention_forward(q, k, v, scale: float, is_causal: bool = False, mask=None, mask_stride_b: int = 0,
                      mask_stride_h: int = 0, return_probs: bool = False, return_lse: bool = False):
    """O = softmax(Q K^T * scale + mask, causal) V for q [B,H,S,D], k [B,H,S,D], v [B,H,S,Dv].

    ``mask`` and its strides follow oracle.forward (additive of q's storage
    dtype, or boolean / uint8 with nonzero = masked; row r of the [B*H*S, S]
    score view reads mask[b*stride_b + h*stride_h + i*S ...]).  ``scale`` is
    used as given (pass the float32 value a kernel sees).  Returns O (fp64),
    then P when ``return_probs``, then the per-row log of the softmax
    denominator when ``return_lse`` (see ``log_sum_exp``).
    """
    Q, K, V = _bhsd(_f64(q), "q"), _bhsd(_f64(k), "k"), _bhsd(_f64(v), "v")
    B, H, S, D = Q.shape
    if K.shape != (B, H, S, D) or V.shape[:3] != (B, H, S):
        raise ValueError("q, k, v must share B, H and S (square attention), q and k the head dim")
    scores = np.matmul(Q, np.swapaxes(K, -1, -2))  # [B, H, S, S]
    if mask is not None and not _is_bool(mask):
        mask = decode(mask)  # an additive mask of the inputs' storage dtype, widened exactly
    P = _softmax_forward(scores.reshape(-1, S), S, scale, is_causal, mask, mask_stride_b, mask_stride_h, H)
    P = P.reshape(B, H, S, S)
    O = np.matmul(P, V)
    out = [O]
    if return_probs:
        out.append(P)
    if return_lse:
        out.append(log_sum_exp(scores, scale, is_causal, mask, mask_stride_b, mask_stride_h))
    return tuple(out) if len(out) > 1 else O


def log_sum_exp(scores, scale: float, is_causal: bool = False, mask=None, mask_stride_b: int = 0,
                mask_stride_h: int = 0):
    """Per query row, log sum_j exp(s_j) of the scores s = scores*scale + mask
    (j > i masked under causal), the log of the softmax denominator: with
    M = max_j s_j it is M + log sum_j exp(s_j - M), and -inf for a row whose
    every score is -inf.  ``scores`` is the fp64 [B, H, S, S] product Q K^T;
    the mask follows oracle.forward (additive, or boolean / uint8 with
    nonzero = masked)."""
    B, H, S, _ = scores.shape
    s = np.asarray(scores, dtype=np.float64) * float(scale)
    if mask is not None:
        m = np.asarray(decode(mask) if not _is_bool(mask) else _bool_np(mask), dtype=np.float64).reshape(-1)
        for b in range(B):
            for h in range(H):
                base = b * mask_stride_b + h * mask_stride_h
                s[b, h] += m[base:base + S * S].reshape(S, S)
    if is_causal:
        s = np.where(np.triu(np.ones((S, S), dtype=bool), 1), -np.inf, s)
    M = s.max(axis=-1)
    live = M > -np.inf
    Mr = np.where(live, M, 0.0)
    tot = np.exp(s - Mr[..., None]).sum(axis=-1)
    return np.where(live, Mr + np.log(np.where(live, tot, 1.0)), -np.inf)


def _is_bool(mask) -> bool:
    try:
        import torch

        if isinstance(mask, torch.Tensor):
            return mask.dtype in (torch.bool, torch.uint8)
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(mask).dtype in (np.bool_, np.uint8)


def _bool_np(mask) -> np.ndarray:
    """A boolean / byte mask as additive fp64 values: -inf where nonzero, else 0."""
    try:
        import torch

        if isinstance(mask, torch.Tensor):
            mask = mask.detach().to("cpu").numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.where(np.asarray(mask).astype(np.uint8) != 0, -np.inf, 0.0)


def attention_backward(q, k, v, d_o, scale: float, is_causal: bool = False, mask=None, mask_stride_b: int = 0,
                       mask_stride_h: int = 0):
    """(dQ, dK, dV) of sum(dO * O) for the forward above, in fp64."""
    Q, K, V = _f64(q), _f64(k), _f64(v)
    dO = _f64(d_o)
    O, P = attention_forward(Q, K, V, scale, is_causal, mask, mask_stride_b, mask_stride_h, return_probs=True)
    B, H, S, _ = Q.shape
    dV = np.matmul(np.swapaxes(P, -1, -2), dO)
    dP = np.matmul(dO, np.swapaxes(V, -1, -2))
    dS = _softmax_backward(P.reshape(-1, S), dP.reshape(-1, S), S, scale).reshape(B, H, S, S)
    dQ = np.matmul(dS, K)
    dK = np.matmul(np.swapaxes(dS, -1, -2), Q)
    return dQ, dK, dV
