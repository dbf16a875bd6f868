"""Seeded synthetic workloads for the fused ScaledMaskSoftmax.

This module only draws inputs (scores, additive masks, upstream gradients) and
describes their shapes; it holds none of the operator's arithmetic, so both the
CUDA path and the fp64 oracle can be fed from it.

The workloads follow the shapes and value distributions of the attention
score tensors on the source pages: a [B,H,S,S] score tensor viewed as
[rows = B*H*S, cols = S] (page "用CUDA自定义融合Softmax算子并封装进PyTorch" §2.3 and
§4.2), scores distributed like QK^T of unit-variance q/k with head dim d_k
(x ~ N(0, d_k)) and scale 1/sqrt(d_k) (same page §1.2), additive key-padding
masks with 0 for kept keys and -10000 or -inf for padding (same page §2.2), and
the causal flag (same page §1.2).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    S: int
    dtype: str                 # "f32" | "f16" | "bf16"
    sigma: float               # x ~ N(0, sigma^2)
    scale: float               # float32 value handed to the kernel
    mask: str                  # "none" | "B1SS" (key padding) | "SS" (random broadcast) | "BHSS" (full, tests)
    is_causal: bool
    backward: bool             # the workload also runs the backward
    seed: int
    pad_fill: float = 0.0      # value of padded / dropped mask entries
    pad_lo: float = 0.5        # key-padding length L_b ~ U[pad_lo*S, S] (integers, inclusive)
    drop_p: float = 0.0        # "SS": probability that an entry is dropped (column 0 never)
    spike_frac: float = 0.0    # fraction of rows that get one +spike_value score
    spike_value: float = 6.0e4
    rows_override: Optional[int] = None  # rows not equal to B*H*S (the width sweep)
    mask_values: str = "zero"  # kept mask entries: "zero" or "normal" (N(0,1), tests only)

    @property
    def rows(self) -> int:
        return self.rows_override if self.rows_override is not None else self.B * self.H * self.S

    @property
    def cols(self) -> int:
        return self.S

    @property
    def torch_dtype(self) -> torch.dtype:
        return DTYPES[self.dtype]

    @property
    def elem_bytes(self) -> int:
        return torch.empty((), dtype=self.torch_dtype).element_size()

    def mask_strides(self):
        """(mask_stride_b, mask_stride_h, heads) of the additive mask."""
        if self.mask == "B1SS":
            return self.S * self.S, 0, self.H
        if self.mask == "BHSS":
            return self.H * self.S * self.S, self.S * self.S, self.H
        return 0, 0, self.H

    def mask_shape(self):
        if self.mask == "B1SS":
            return (self.B, 1, self.S, self.S)
        if self.mask == "SS":
            return (min(self.S, self.rows), self.S)
        if self.mask == "BHSS":
            return (self.B, self.H, self.S, self.S)
        return None


def _f32(v: float) -> float:
    return float(torch.tensor(v, dtype=torch.float32).item())


_SWEEP_S = (128, 256, 512, 1000, 1024, 2048, 4099, 8192, 16384)

WORKLOADS = {
    # B=1 H=2 S=64 fp32, causal, no mask (small enough for the oracle in milliseconds)
    "tiny_causal_f32": Workload("tiny_causal_f32", 1, 2, 64, "f32", 8.0, 0.125, "none", True, False, 1),
    # B=8 H=32 S=1024 fp32, [B,1,S,S] key padding with -10000, L_b ~ U[S/2, S]
    "keypad_f32_s1024": Workload("keypad_f32_s1024", 8, 32, 1024, "f32", 8.0, 0.125, "B1SS", False, True, 2,
                                 pad_fill=-10000.0, pad_lo=0.5),
    # B=4 H=32 S=2048 fp16, causal, 1% of rows carry a +6e4 spike at a kept column
    "causal_spike_f16_s2048": Workload("causal_spike_f16_s2048", 4, 32, 2048, "f16", 8.0, 0.125, "none", True, True,
                                       3, spike_frac=0.01),
    # B=4 H=32 S=4096 bf16 (d_k=128), [B,1,S,S] key padding with -inf, L_b ~ U[S/4, S], causal
    "keypad_causal_bf16_s4096": Workload("keypad_causal_bf16_s4096", 4, 32, 4096, "bf16", 11.3,
                                         _f32(1.0 / math.sqrt(128.0)), "B1SS", True, True, 4,
                                         pad_fill=-math.inf, pad_lo=0.25),
}
for _dt in ("f16", "f32"):
    for _S in _SWEEP_S:
        _name = f"sweep_{_dt}_s{_S}"
        # rows = 2^26 // S, [S,S] mask with 10% of entries at -inf (column 0 never masked)
        WORKLOADS[_name] = Workload(_name, 1, 1, _S, _dt, 8.0, 0.125, "SS", False, False, 5,
                                    pad_fill=-math.inf, drop_p=0.1, rows_override=(1 << 26) // _S)


def scaled(w: Workload, B: int = None, H: int = None, S: int = None, rows: int = None) -> Workload:
    """The same distributions on a smaller shape (parity tests)."""
    kw = {}
    if B is not None:
        kw["B"] = B
    if H is not None:
        kw["H"] = H
    if S is not None:
        kw["S"] = S
    if rows is not None:
        kw["rows_override"] = rows
    elif w.rows_override is not None:
        kw["rows_override"] = None
    return dataclasses.replace(w, name=w.name + "_scaled", **kw)


def make_inputs(w: Workload, device="cpu", with_dy: Optional[bool] = None):
    """Draw x, the additive mask and dy for workload ``w`` on ``device``.

    Returns a dict with x [rows, cols], mask (None or its broadcast shape),
    dy (or None), the mask broadcast description, and for key-padding
    workloads the padding as per-batch key lengths (int32 [B], else None).  Draws are seeded by
    ``w.seed``; small integer choices (padding lengths, spike rows/columns)
    are drawn on the CPU so they do not depend on the device.
    """
    if with_dy is None:
        with_dy = w.backward
    dt = w.torch_dtype
    dev = torch.device(device)
    g_dev = torch.Generator(device=dev).manual_seed(w.seed)
    g_cpu = torch.Generator().manual_seed(w.seed + 1000)
    rows, S = w.rows, w.S

    x = torch.randn(rows, S, generator=g_dev, device=dev, dtype=torch.float32).mul_(w.sigma).to(dt)

    if w.spike_frac > 0:
        n_spike = max(1, int(round(rows * w.spike_frac)))
        r_idx = torch.randperm(rows, generator=g_cpu)[:n_spike]
        q = r_idx % S
        limit = (q + 1) if w.is_causal else torch.full_like(q, S)
        c_idx = (torch.rand(n_spike, generator=g_cpu, dtype=torch.float64) * limit.double()).floor().long()
        c_idx = torch.minimum(c_idx, limit - 1)
        x[r_idx.to(dev), c_idx.to(dev)] = torch.tensor(w.spike_value, dtype=dt, device=dev)

    mask = None
    key_lengths = None
    if w.mask == "B1SS":
        lo = int(math.ceil(w.pad_lo * S))
        L = torch.randint(lo, S + 1, (w.B,), generator=g_cpu)
        key_lengths = L.to(torch.int32).to(dev)  # the same padding as per-batch key lengths
        cols_idx = torch.arange(S, device=dev)
        keep = cols_idx[None, :] < L.to(dev)[:, None]  # [B, S]
        mrow = torch.where(keep, torch.tensor(0.0, device=dev), torch.tensor(w.pad_fill, device=dev))
        mask = mrow[:, None, None, :].expand(w.B, 1, S, S).to(dt).contiguous()
    elif w.mask == "BHSS":
        drop = torch.rand(w.B, w.H, S, S, generator=g_dev, device=dev) < w.drop_p
        drop[..., 0] = False
        vals = torch.randn(w.B, w.H, S, S, generator=g_dev, device=dev) if w.mask_values == "normal" else \
            torch.zeros(w.B, w.H, S, S, device=dev)
        mask = torch.where(drop, torch.tensor(w.pad_fill, device=dev), vals).to(dt)
    elif w.mask == "SS":
        # only the first min(rows, S) query rows of an [S,S] mask are ever read
        # (row r reads mask row r mod S), so only those are materialised
        drop = torch.rand(min(S, rows), S, generator=g_dev, device=dev) < w.drop_p
        drop[:, 0] = False
        mask = torch.where(drop, torch.tensor(w.pad_fill, device=dev), torch.tensor(0.0, device=dev)).to(dt)
        if w.mask_values == "normal":  # finite additive values as well as dropped entries
            vals = torch.randn(min(S, rows), S, generator=g_dev, device=dev)
            mask = torch.where(drop, torch.tensor(w.pad_fill, device=dev), vals).to(dt)
            mask[:, 0] = 0

    dy = None
    if with_dy:
        dy = torch.randn(rows, S, generator=g_dev, device=dev, dtype=torch.float32).to(dt)

    sb, sh, heads = w.mask_strides()
    return {"x": x, "mask": mask, "dy": dy, "mask_stride_b": sb, "mask_stride_h": sh, "heads": heads,
            "key_lengths": key_lengths}



def attention_inputs(B: int, H: int, S: int, D: int, dtype: str, seed: int, device="cpu", sigma: float = 1.0,
                     with_do: bool = False):
    """Seeded q, k, v (and dO) of a [B, H, S, D] attention step: entries
    ~ N(0, sigma^2) for q and k (so q.k ~ N(0, D sigma^4), the score
    distribution the softmax workloads model with x ~ N(0, d_k)), v and dO
    ~ N(0, 1), drawn in fp32 on ``device`` and rounded to ``dtype``."""
    dt = DTYPES[dtype]
    g = torch.Generator(device=torch.device(device)).manual_seed(seed)
    shape = (B, H, S, D)
    q = (torch.randn(shape, generator=g, device=device) * sigma).to(dt)
    k = (torch.randn(shape, generator=g, device=device) * sigma).to(dt)
    v = torch.randn(shape, generator=g, device=device).to(dt)
    d_o = torch.randn(shape, generator=g, device=device).to(dt) if with_do else None
    return q, k, v, d_o
