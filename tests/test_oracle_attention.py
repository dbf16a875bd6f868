"""Pins of the fp64 attention oracle (oracle/attention.py): softmax(Q K^T * scale
+ mask, causal) V and its gradient, against what does not come from the
oracle itself: torch's scaled_dot_product_attention in fp64 (a library special
case), closed forms (zero queries give key means, a single kept key selects
its value row, V = I returns the probabilities), the fully masked row rule,
central finite differences, and fp64 autograd through torch's own ops."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as A

F = torch.nn.functional


def _qkv(B, H, S, D, Dv, seed, dtype=torch.float64, sigma=1.0):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(B, H, S, D, generator=g, dtype=torch.float64) * sigma).to(dtype)
    k = (torch.randn(B, H, S, D, generator=g, dtype=torch.float64) * sigma).to(dtype)
    v = torch.randn(B, H, S, Dv, generator=g, dtype=torch.float64).to(dtype)
    return q, k, v


@pytest.mark.parametrize("dtype", [torch.float64, torch.float32, torch.float16, torch.bfloat16])
@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_sdpa(dtype, causal):
    q, k, v = _qkv(2, 3, 17, 8, 5, 1, dtype)
    scale = float(np.float32(1 / math.sqrt(8)))
    O = A.attention_forward(q, k, v, scale, causal)
    ref = F.scaled_dot_product_attention(q.double(), k.double(), v.double(), is_causal=causal, scale=scale)
    assert np.abs(O - ref.numpy()).max() < 1e-13


@pytest.mark.parametrize("layout", ["SS", "B1SS", "BHSS"])
@pytest.mark.parametrize("causal", [False, True])
def test_additive_mask_layouts_match_torch_sdpa(layout, causal):
    B, H, S = 2, 3, 11
    q, k, v = _qkv(B, H, S, 4, 6, 2)
    g = torch.Generator().manual_seed(3)
    shape = {"SS": (S, S), "B1SS": (B, 1, S, S), "BHSS": (B, H, S, S)}[layout]
    mask = torch.randn(shape, generator=g, dtype=torch.float64) * 3  # finite: no fully masked row
    sb, sh = {"SS": (0, 0), "B1SS": (S * S, 0), "BHSS": (H * S * S, S * S)}[layout]
    O = A.attention_forward(q, k, v, 0.25, causal, mask, sb, sh)
    full = mask.expand(B, H, S, S)
    if causal:
        full = full.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), -math.inf)
    ref = F.scaled_dot_product_attention(q, k, v, attn_mask=full, scale=0.25)
    assert np.abs(O - ref.numpy()).max() < 1e-13


def test_zero_queries_give_key_means():
    # every score is 0: O_i is the mean of the kept value rows (all of them, or
    # the prefix j <= i under causal)
    B, H, S, Dv = 1, 2, 9, 3
    _, k, v = _qkv(B, H, S, 4, Dv, 4)
    q = torch.zeros(B, H, S, 4, dtype=torch.float64)
    O = A.attention_forward(q, k, v, 0.5, False)
    assert np.allclose(O, v.mean(dim=2, keepdim=True).expand(B, H, S, Dv).numpy(), rtol=0, atol=1e-15)
    Oc = A.attention_forward(q, k, v, 0.5, True)
    prefix = torch.cumsum(v, dim=2) / torch.arange(1, S + 1, dtype=torch.float64).view(1, 1, S, 1)
    assert np.allclose(Oc, prefix.numpy(), rtol=0, atol=1e-15)


def test_single_kept_key_selects_its_value_row():
    B, H, S = 1, 1, 7
    q, k, v = _qkv(B, H, S, 5, 4, 5)
    keep = [3, 0, 6, 6, 1, 2, 5]  # row i keeps only key keep[i]
    mask = torch.ones(S, S, dtype=torch.bool)
    for i, j in enumerate(keep):
        mask[i, j] = False
    O = A.attention_forward(q, k, v, 0.7, False, mask)
    assert np.array_equal(O[0, 0], v[0, 0, keep].numpy())


def test_identity_values_return_the_probabilities():
    B, H, S = 2, 2, 6
    q, k, _ = _qkv(B, H, S, 3, S, 6)
    eye = torch.eye(S, dtype=torch.float64).expand(B, H, S, S).contiguous()
    O, P = A.attention_forward(q, k, eye, 0.9, True, return_probs=True)
    assert np.array_equal(O, P)
    assert np.allclose(P.sum(-1), 1.0, rtol=0, atol=1e-15)
    assert np.all(P[..., np.triu_indices(S, 1)[0], np.triu_indices(S, 1)[1]] == 0.0)


def test_fully_masked_row_is_zero_with_zero_gradient():
    B, H, S = 1, 2, 5
    q, k, v = _qkv(B, H, S, 3, 4, 7)
    mask = torch.zeros(S, S, dtype=torch.bool)
    mask[2, :] = True  # query 2 keeps no key
    O = A.attention_forward(q, k, v, 0.5, False, mask)
    assert np.all(O[:, :, 2] == 0.0)
    d_o = torch.randn(B, H, S, 4, generator=torch.Generator().manual_seed(8), dtype=torch.float64)
    dQ, dK, dV = A.attention_backward(q, k, v, d_o, 0.5, False, mask)
    assert np.all(dQ[:, :, 2] == 0.0)
    # query 2 contributes nothing to dK / dV: zeroing its dO row leaves them unchanged
    d_o2 = d_o.clone()
    d_o2[:, :, 2] = 0
    _, dK2, dV2 = A.attention_backward(q, k, v, d_o2, 0.5, False, mask)
    assert np.array_equal(dK, dK2) and np.array_equal(dV, dV2)


def test_backward_finite_differences():
    B, H, S, D, Dv = 1, 1, 4, 3, 2
    q, k, v = _qkv(B, H, S, D, Dv, 9)
    d_o = torch.randn(B, H, S, Dv, generator=torch.Generator().manual_seed(10), dtype=torch.float64)
    scale = 0.6
    mask = torch.tensor([[0.0, -1.0, 0.5, 0.0]] * S, dtype=torch.float64)
    dQ, dK, dV = A.attention_backward(q, k, v, d_o, scale, True, mask)

    def loss(qq, kk, vv):
        return float(np.sum(A.attention_forward(qq, kk, vv, scale, True, mask) * d_o.numpy()))

    h = 1e-6
    for name, t, grad in (("q", q, dQ), ("k", k, dK), ("v", v, dV)):
        num = np.zeros(t.shape)
        for idx in np.ndindex(*t.shape):
            tp, tm = t.clone(), t.clone()
            tp[idx] += h
            tm[idx] -= h
            args_p = {"q": q, "k": k, "v": v, name: tp}
            args_m = {"q": q, "k": k, "v": v, name: tm}
            num[idx] = (loss(args_p["q"], args_p["k"], args_p["v"]) - loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * h)
        err = np.abs(num - grad).max() / max(np.abs(grad).max(), 1e-12)
        assert err < 1e-6, (name, err)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_torch_autograd(causal):
    B, H, S, D, Dv = 2, 2, 13, 4, 5
    q, k, v = _qkv(B, H, S, D, Dv, 11)
    d_o = torch.randn(B, H, S, Dv, generator=torch.Generator().manual_seed(12), dtype=torch.float64)
    mask = torch.rand(B, 1, S, S, generator=torch.Generator().manual_seed(13)) < 0.2
    mask[..., 0] = False  # every row keeps key 0
    scale = float(np.float32(0.35))
    dQ, dK, dV = A.attention_backward(q, k, v, d_o, scale, causal, mask, S * S, 0)
    qt, kt, vt = (t.clone().requires_grad_(True) for t in (q, k, v))
    s = torch.matmul(qt, kt.transpose(-1, -2)) * scale
    s = s.masked_fill(mask.expand(B, H, S, S), -math.inf)
    if causal:
        s = s.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), -math.inf)
    o = torch.matmul(torch.softmax(s, dim=-1), vt)
    o.backward(d_o)
    for mine, ref in ((dQ, qt.grad), (dK, kt.grad), (dV, vt.grad)):
        assert np.abs(mine - ref.numpy()).max() < 1e-12


def test_inputs_are_decoded_exactly():
    # fp16 / bf16 inputs are widened exactly: the same values given as fp64 give the same result bit for bit
    q, k, v = _qkv(1, 2, 8, 4, 3, 14, torch.bfloat16, sigma=4.0)
    a = A.attention_forward(q, k, v, 0.5, True)
    b = A.attention_forward(q.double(), k.double(), v.double(), 0.5, True)
    assert np.array_equal(a, b)
    assert np.array_equal(oracle.decode(q).reshape(q.shape), q.double().numpy())


# ------------------------------------------------------------- log-sum-exp ---

@pytest.mark.parametrize("layout", ["none", "SS", "B1SS", "BHSS", "bool"])
@pytest.mark.parametrize("causal", [False, True])
def test_lse_matches_torch_logsumexp(layout, causal):
    """The per-row log of the softmax denominator against torch.logsumexp of
    the same masked scores (fp64, a library routine)."""
    B, H, S = 2, 3, 13
    q, k, v = _qkv(B, H, S, 8, 4, 21)
    g = torch.Generator().manual_seed(22)
    shape = {"none": None, "SS": (S, S), "B1SS": (B, 1, S, S), "BHSS": (B, H, S, S), "bool": (B, 1, S, S)}[layout]
    sb, sh = {"none": (0, 0), "SS": (0, 0), "B1SS": (S * S, 0), "BHSS": (H * S * S, S * S),
              "bool": (S * S, 0)}[layout]
    mask = None
    full = torch.zeros(B, H, S, S, dtype=torch.float64)
    if layout == "bool":
        mask = torch.rand(shape, generator=g) < 0.3
        mask[..., 0] = False
        full = torch.zeros(shape, dtype=torch.float64).masked_fill(mask, -math.inf).expand(B, H, S, S)
    elif shape is not None:
        mask = torch.randn(shape, generator=g, dtype=torch.float64) * 2
        full = mask.expand(B, H, S, S)
    scale = 0.3
    O, lse = A.attention_forward(q, k, v, scale, causal, mask, sb, sh, return_lse=True)
    s = torch.matmul(q, k.transpose(-1, -2)) * scale + full
    if causal:
        s = s.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), -math.inf)
    ref = torch.logsumexp(s, -1).numpy()
    assert np.abs(lse - ref).max() < 1e-12


def test_lse_closed_forms():
    # zero queries: every kept score is 0, so lse = log(number of kept keys):
    # log S without causal, log(i + 1) for row i under causal; a row with every
    # key masked is -inf
    B, H, S = 1, 2, 6
    _, k, v = _qkv(B, H, S, 4, 3, 23)
    q = torch.zeros(B, H, S, 4, dtype=torch.float64)
    _, lse = A.attention_forward(q, k, v, 1.0, False, return_lse=True)
    assert np.allclose(lse, math.log(S), rtol=0, atol=1e-15)
    _, lse_c = A.attention_forward(q, k, v, 1.0, True, return_lse=True)
    assert np.allclose(lse_c, np.log(np.arange(1, S + 1))[None, None, :], rtol=0, atol=1e-15)
    mask = torch.zeros(S, S, dtype=torch.bool)
    mask[2, :] = True
    _, lse_m = A.attention_forward(q, k, v, 1.0, False, mask, return_lse=True)
    assert np.all(np.isneginf(lse_m[:, :, 2]))
    assert np.allclose(np.delete(lse_m, 2, axis=2), math.log(S), rtol=0, atol=1e-15)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_additive_mask_of_the_storage_dtype(dtype):
    """An additive mask stored in q's 16-bit dtype (the layout the kernels
    take) is widened exactly: the result equals torch SDPA with that mask
    converted to fp64 by torch."""
    B, H, S = 2, 2, 9
    q, k, v = _qkv(B, H, S, 8, 3, 31, dtype)
    g = torch.Generator().manual_seed(32)
    mask = (torch.randn(B, 1, S, S, generator=g) * 3).to(dtype)
    mask[0, 0, 3, 5] = -math.inf
    O, lse = A.attention_forward(q, k, v, 0.4, False, mask, S * S, 0, return_lse=True)
    full = mask.double().expand(B, H, S, S)
    ref = F.scaled_dot_product_attention(q.double(), k.double(), v.double(), attn_mask=full, scale=0.4)
    assert np.abs(O - ref.numpy()).max() < 1e-13
    s = torch.matmul(q.double(), k.double().transpose(-1, -2)) * 0.4 + full
    assert np.abs(lse - torch.logsumexp(s, -1).numpy()).max() < 1e-12
