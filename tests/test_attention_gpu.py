"""GPU parity of the fused attention step (tensor-core kernels through the C
ABI) against the fp64 oracle of oracle/attention.py.

Tolerance (the pages state none for this step; derived from the arithmetic):
Q K^T is exact products summed in fp32, the softmax runs in fp32, P is
rounded once to the 16-bit dtype (relative u/2) and O once more (relative
u/2), with u the unit roundoff (2^-8 bf16, 2^-11 fp16), so
    |O - O_ref| <= 2u (|O_ref| + (P |V|)) + S 2^-24 max|V| [fp16] + 1e-6
elementwise, where P |V| is the oracle's probabilities times |V| and the
fp16 term covers probabilities below fp16's normal range.  lse is fp32:
|lse - lse_ref| <= 1e-3 max(1, |lse_ref|).  Rows whose every key is masked
give O = 0 exactly and lse = -inf.
"""
import math

import numpy as np
import pytest
import torch

import scaled_masked_softmax_gb300 as sms
from oracle import attention as A
from scaled_masked_softmax_gb300 import workloads

pytestmark = pytest.mark.gpu

TD = {"f16": torch.float16, "bf16": torch.bfloat16}
UNIT = {"f16": 2.0 ** -11, "bf16": 2.0 ** -8}


def _check(o, lse, q, k, v, dt, scale, causal, mask=None, sb=0, sh=0, what=""):
    torch.cuda.synchronize()
    assert sms.sms_device_error(torch.cuda.current_stream().cuda_stream) == 0
    qc, kc, vc = q.cpu(), k.cpu(), v.cpu()
    mc = mask.cpu() if mask is not None else None
    O, P, L = A.attention_forward(qc, kc, vc, scale, causal, mc, sb, sh, return_probs=True, return_lse=True)
    Vabs = np.abs(vc.double().numpy())
    S = q.shape[2]
    bound = 2 * UNIT[dt] * (np.abs(O) + np.matmul(P, Vabs)) + 1e-6
    if dt == "f16":
        bound += S * 2.0 ** -24 * float(Vabs.max())
    og = o.double().cpu().numpy()
    assert np.all(np.isfinite(og)), f"{what}: non-finite output"
    excess = np.abs(og - O) - bound
    assert float(excess.max()) <= 0, f"{what}: |O - O_ref| exceeds the bound by {float(excess.max()):.3e} " \
                                     f"(max err {float(np.abs(og - O).max()):.3e})"
    dead = np.isneginf(L)
    assert np.all(og[dead] == 0.0), f"{what}: fully masked rows must be 0"
    lg = lse.double().cpu().numpy()
    assert np.array_equal(np.isneginf(lg), dead), f"{what}: -inf lse rows differ"
    live = ~dead
    err = np.abs(lg[live] - L[live]) / np.maximum(1.0, np.abs(L[live]))
    assert err.size == 0 or float(err.max()) <= 1e-3, f"{what}: lse error {float(err.max()):.3e}"


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("S", [1, 7, 64, 128, 129, 200, 256, 300])
@pytest.mark.parametrize("causal", [False, True])
def test_attention_forward_shapes(dt, D, S, causal):
    B, H = 2, 3
    q, k, v, _ = workloads.attention_inputs(B, H, S, D, dt, seed=S * 7 + D, device="cuda")
    scale = float(np.float32(1.0 / math.sqrt(D)))
    o, lse = sms.attention_forward(q, k, v, None, scale, causal, return_lse=True)
    _check(o, lse, q, k, v, dt, scale, causal, what=f"{dt} D={D} S={S} causal={causal}")


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("layout", ["SS", "B1SS", "BHSS", "bool_SS", "bool_B1SS"])
@pytest.mark.parametrize("causal", [False, True])
def test_attention_forward_masks(dt, layout, causal):
    B, H, S, D = 2, 3, 200, 64
    q, k, v, _ = workloads.attention_inputs(B, H, S, D, dt, seed=91, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(92)
    kind = layout.split("_")[-1]
    shape = {"SS": (S, S), "B1SS": (B, 1, S, S), "BHSS": (B, H, S, S)}[kind]
    sb, sh = {"SS": (0, 0), "B1SS": (S * S, 0), "BHSS": (H * S * S, S * S)}[kind]
    drop = torch.rand(shape, generator=g, device="cuda") < 0.2
    drop[..., 0] = False
    if layout.startswith("bool"):
        mask = drop.clone()
        mask.view(-1, S)[5] = True  # one query row with every key masked
    else:
        mask = torch.where(drop, torch.tensor(-math.inf, device="cuda"),
                           torch.randn(shape, generator=g, device="cuda")).to(TD[dt])
        mask.view(-1, S)[5] = -math.inf
    o, lse = sms.attention_forward(q, k, v, mask, 0.125, causal, return_lse=True)
    _check(o, lse, q, k, v, dt, 0.125, causal, mask, sb, sh, what=f"{dt} {layout} causal={causal}")


@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_attention_forward_wide_scores(dt):
    """q, k ~ N(0, 3^2): scores spread over hundreds, the running max grows
    by more than 2^8 between key blocks, and the output accumulator is
    rescaled on the way."""
    B, H, S, D = 1, 2, 640, 128
    q, k, v, _ = workloads.attention_inputs(B, H, S, D, dt, seed=5, device="cuda", sigma=3.0)
    o, lse = sms.attention_forward(q, k, v, None, 0.5, False, return_lse=True)
    _check(o, lse, q, k, v, dt, 0.5, False, what=f"{dt} wide scores")


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("causal", [False, True])
def test_attention_forward_long(dt, causal):
    """Several hundred CTAs and 16 key blocks per query tile (d_k = 128)."""
    B, H, S, D = 1, 4, 2048, 128
    q, k, v, _ = workloads.attention_inputs(B, H, S, D, dt, seed=17, device="cuda")
    scale = float(np.float32(1.0 / math.sqrt(D)))
    o, lse = sms.attention_forward(q, k, v, None, scale, causal, return_lse=True)
    _check(o, lse, q, k, v, dt, scale, causal, what=f"{dt} S={S} causal={causal}")


def test_attention_forward_rejects():
    q, k, v, _ = workloads.attention_inputs(1, 1, 16, 64, "bf16", seed=1, device="cuda")
    with pytest.raises(sms.SmsError) as e:
        sms.sms_attention_forward(q.float().data_ptr(), k.data_ptr(), v.data_ptr(), None, 0, 0, 0, 0, q.data_ptr(),
                                  None, 1, 1, 16, 64, 0.1, False, sms.SMS_F32, 0)
    assert e.value.status == 2
    with pytest.raises(sms.SmsError) as e:
        sms.sms_attention_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), None, 0, 0, 0, 0, q.data_ptr(), None, 1, 1,
                                  16, 64, 0.1, False, sms.SMS_BF16, 0)
    assert e.value.status == 1  # o aliases q


# ------------------------------------------------------------------ backward ---
# Tolerance of dQ, dK, dV (the pages state none; derived from the arithmetic):
# P and dS enter the MMAs rounded to the 16-bit dtype, delta comes from the
# stored 16-bit O, every gradient is rounded once.  With
#   A_ij = sum_d |dO_id| |V_jd|,  delta'_i = sum_j P_ij A_ij,
#   G = P * (A + delta'),          (first-order size of the terms of dS / scale)
#   M_dV = P^T |dO|, M_dQ = scale G |K|, M_dK = scale G^T |Q|
# the bound is |X - X_ref| <= 6u M_X + u |X_ref| + 1e-5 max M_X, plus for fp16
# S 2^-23 (1 + scale max(A + delta')) max(|Q|, |K|, |dO|) for probabilities and
# gradients below fp16's normal range.

def _check_bwd(dq, dk, dv, q, k, v, d_o, dt, scale, causal, mask=None, sb=0, sh=0, what=""):
    torch.cuda.synchronize()
    assert sms.sms_device_error(torch.cuda.current_stream().cuda_stream) == 0
    qc, kc, vc, gc = q.cpu(), k.cpu(), v.cpu(), d_o.cpu()
    mc = mask.cpu() if mask is not None else None
    dQ, dK, dV = A.attention_backward(qc, kc, vc, gc, scale, causal, mc, sb, sh)
    _, P = A.attention_forward(qc, kc, vc, scale, causal, mc, sb, sh, return_probs=True)
    Q64, K64, V64, G64 = (np.abs(t.double().numpy()) for t in (qc, kc, vc, gc))
    Am = np.matmul(G64, np.swapaxes(V64, -1, -2))
    dlt = np.sum(P * Am, axis=-1, keepdims=True)
    G = P * (Am + dlt)
    mags = {"dV": np.matmul(np.swapaxes(P, -1, -2), G64), "dQ": abs(scale) * np.matmul(G, K64),
            "dK": abs(scale) * np.matmul(np.swapaxes(G, -1, -2), Q64)}
    u = UNIT[dt]
    S = q.shape[2]
    extra = 0.0
    if dt == "f16":
        extra = S * 2.0 ** -23 * (1 + abs(scale) * float((Am + dlt).max())) * max(Q64.max(), K64.max(), G64.max())
    for name, got, ref in (("dQ", dq, dQ), ("dK", dk, dK), ("dV", dv, dV)):
        g = got.double().cpu().numpy()
        assert np.all(np.isfinite(g)), f"{what} {name}: non-finite"
        M = mags[name]
        bound = 6 * u * M + u * np.abs(ref) + 1e-5 * float(M.max()) + extra + 1e-7
        excess = np.abs(g - ref) - bound
        assert float(excess.max()) <= 0, f"{what} {name}: error exceeds the bound by {float(excess.max()):.3e} " \
                                         f"(max err {float(np.abs(g - ref).max()):.3e}, max ref {float(np.abs(ref).max()):.3e})"


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("S", [1, 7, 128, 129, 200, 256, 300])
@pytest.mark.parametrize("causal", [False, True])
def test_attention_backward_shapes(dt, D, S, causal):
    B, H = 2, 2
    q, k, v, d_o = workloads.attention_inputs(B, H, S, D, dt, seed=S * 3 + D + 1, device="cuda", with_do=True)
    scale = float(np.float32(1.0 / math.sqrt(D)))
    o, lse = sms.attention_forward(q, k, v, None, scale, causal, return_lse=True)
    dq, dk, dv = sms.attention_backward(q, k, v, o, lse, d_o, None, scale, causal)
    _check_bwd(dq, dk, dv, q, k, v, d_o, dt, scale, causal, what=f"{dt} D={D} S={S} causal={causal}")


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("layout", ["SS", "B1SS", "BHSS", "bool_B1SS"])
@pytest.mark.parametrize("causal", [False, True])
def test_attention_backward_masks(dt, layout, causal):
    B, H, S, D = 2, 2, 200, 64
    q, k, v, d_o = workloads.attention_inputs(B, H, S, D, dt, seed=71, device="cuda", with_do=True)
    g = torch.Generator(device="cuda").manual_seed(72)
    kind = layout.split("_")[-1]
    shape = {"SS": (S, S), "B1SS": (B, 1, S, S), "BHSS": (B, H, S, S)}[kind]
    sb, sh = {"SS": (0, 0), "B1SS": (S * S, 0), "BHSS": (H * S * S, S * S)}[kind]
    drop = torch.rand(shape, generator=g, device="cuda") < 0.2
    drop[..., 0] = False
    if layout.startswith("bool"):
        mask = drop.clone()
        mask.view(-1, S)[5] = True
    else:
        mask = torch.where(drop, torch.tensor(-math.inf, device="cuda"),
                           torch.randn(shape, generator=g, device="cuda")).to(TD[dt])
        mask.view(-1, S)[5] = -math.inf
    o, lse = sms.attention_forward(q, k, v, mask, 0.125, causal, return_lse=True)
    dq, dk, dv = sms.attention_backward(q, k, v, o, lse, d_o, mask, 0.125, causal)
    _check_bwd(dq, dk, dv, q, k, v, d_o, dt, 0.125, causal, mask, sb, sh, what=f"{dt} {layout} causal={causal}")


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("causal", [False, True])
def test_attention_backward_long(dt, causal):
    B, H, S, D = 1, 2, 1024, 128
    q, k, v, d_o = workloads.attention_inputs(B, H, S, D, dt, seed=19, device="cuda", with_do=True)
    scale = float(np.float32(1.0 / math.sqrt(D)))
    o, lse = sms.attention_forward(q, k, v, None, scale, causal, return_lse=True)
    dq, dk, dv = sms.attention_backward(q, k, v, o, lse, d_o, None, scale, causal)
    _check_bwd(dq, dk, dv, q, k, v, d_o, dt, scale, causal, what=f"{dt} S={S} causal={causal}")


def test_fused_attention_autograd():
    B, H, S, D = 2, 2, 160, 64
    q, k, v, d_o = workloads.attention_inputs(B, H, S, D, "bf16", seed=81, device="cuda", with_do=True)
    mask = torch.zeros(B, 1, S, S, dtype=torch.bool, device="cuda")
    mask[1, :, :, 100:] = True  # key padding of the second batch
    qg, kg, vg = (t.clone().requires_grad_(True) for t in (q, k, v))
    o = sms.fused_attention(qg, kg, vg, mask, 0.125, True)
    o.backward(d_o)
    _check(o.detach(), sms.attention_forward(q, k, v, mask, 0.125, True, return_lse=True)[1], q, k, v, "bf16", 0.125,
           True, mask, S * S, 0, what="autograd forward")
    _check_bwd(qg.grad, kg.grad, vg.grad, q, k, v, d_o, "bf16", 0.125, True, mask, S * S, 0, what="autograd")
