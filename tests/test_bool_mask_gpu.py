"""GPU parity of the boolean-mask forward (sms_forward_bool).

The page "用CUDA自定义融合Softmax算子并封装进PyTorch" §2.2 builds the additive
mask from a boolean one as mask * (-inf); the kernels read the boolean bytes
directly.  Each case checks the result against the fp64 oracle run on the
boolean mask (nonzero = masked), and bit for bit against the same kernel
family run with the additive mask that §2.2 would build (-inf where masked,
0 elsewhere).  Widths span lane shapes, ragged tails and misaligned mask rows;
layouts cover [S,S], [B,1,S,S] and [B,H,S,S]; fully masked rows give zeros.
"""
import math

import pytest
import torch

import oracle
import scaled_masked_softmax_gb300 as sms
from scaled_masked_softmax_gb300 import workloads
from tests import helpers as H

pytestmark = pytest.mark.gpu

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
WIDTHS = [1, 3, 8, 13, 33, 100, 128, 129, 500, 1000, 1024, 1025, 2049, 3333, 4099, 8192, 12345, 20000]


def _additive(mask_b, dtype):
    z = torch.zeros(mask_b.shape, dtype=torch.float32, device=mask_b.device)
    return z.masked_fill(mask_b != 0, -math.inf).to(dtype)


def _mask(shape, p, seed, kind="bool"):
    """Seeded byte mask: P(masked) = p, column 0 kept, query row 1 (where it
    exists) fully masked; kind "u8" stores 0 / 1 / 255 (any nonzero masks)."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    m = torch.rand(shape, generator=g, device="cuda") < p
    m[..., 0] = False
    if shape[-2] > 1:
        m[..., 1, :] = True
    if kind == "bool":
        return m
    v = torch.randint(1, 256, shape, generator=g, device="cuda", dtype=torch.int32)
    return torch.where(m, v, torch.zeros_like(v)).to(torch.uint8)


def _run(path, fn):
    with H.forced_path(path):
        try:
            out = fn()
        except sms.SmsError as e:
            if e.status == 2:
                pytest.skip(f"{path} path does not take this shape")
            raise
        taken = sms.sms_last_path()
    torch.cuda.synchronize()
    assert sms.sms_device_error(torch.cuda.current_stream().cuda_stream) == 0
    if path != "auto":
        assert taken == H.PATHS[path]
    return out, taken


@pytest.mark.parametrize("path", ["auto", "warp", "stream", "ring", "cta", "online"])
@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("S", WIDTHS)
def test_bool_mask_widths(S, dt, path):
    causal = WIDTHS.index(S) % 2 == 1
    rows = max(3, min(700, 8_000_000 // S))
    w = workloads.Workload(f"b_{S}", 1, 1, S, dt, 8.0, 0.125, "none", causal, False, 61, rows_override=rows)
    x = workloads.make_inputs(w, device="cuda")["x"]
    nq = min(S, rows)
    mb = _mask((nq, S), 0.15, 62 + S, kind="u8" if S % 3 == 0 else "bool")
    ma = _additive(mb, DTYPES[dt])
    y_bool, taken = _run(path, lambda: H.raw_forward_bool(x, mb, 0, 0, 1, w))
    y_add, taken_add = _run(path, lambda: H.raw_forward(dict(x=x, mask=ma, mask_stride_b=0, mask_stride_h=0,
                                                             heads=1), w))
    if taken == taken_add:
        assert torch.equal(y_bool, y_add), f"{path} S={S} {dt}: boolean and additive -inf masks differ"
    y_ref = oracle.forward(x.cpu(), S, w.scale, causal, mb.cpu())
    H.check_forward(H.to_np64(y_bool), y_ref, DTYPES[dt], f"{path} bool S={S} {dt} causal={causal}")
    if rows > 1 and S > 1:
        assert torch.all(y_bool[1] == 0), "a fully masked row must be zero"


@pytest.mark.parametrize("path", ["auto", "warp", "stream", "ring", "cta", "online"])
@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("kind", ["SS", "B1SS", "BHSS"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S", [7, 100, 1000])
def test_bool_mask_layouts(S, causal, kind, dt, path):
    B, Hh = 2, 3
    w = workloads.Workload(f"bl_{S}", B, Hh, S, dt, 8.0, 0.125, "none", causal, False, 63)
    x = workloads.make_inputs(w, device="cuda")["x"]
    shape = {"SS": (S, S), "B1SS": (B, 1, S, S), "BHSS": (B, Hh, S, S)}[kind]
    sb, sh, heads = sms.functional.mask_layout((B, Hh, S, S), shape)
    mb = _mask(shape, 0.3, 64 + S)
    y, taken = _run(path, lambda: H.raw_forward_bool(x, mb.contiguous(), sb, sh, heads, w))
    y_add, taken_add = _run(path, lambda: H.raw_forward(dict(x=x, mask=_additive(mb, DTYPES[dt]), mask_stride_b=sb,
                                                             mask_stride_h=sh, heads=heads), w))
    if taken == taken_add:
        assert torch.equal(y, y_add)
    y_ref = oracle.forward(x.cpu(), S, w.scale, causal, mb.cpu(), sb, sh, heads)
    H.check_forward(H.to_np64(y), y_ref, DTYPES[dt], f"{path} bool {kind} S={S} {dt} causal={causal}")


def test_bool_mask_on_the_cta_path():
    """The staged CTA family stages the mask bytes with the scores: its rows
    (fp32, 8193..16384 columns) take it with a boolean mask too, bit-equal to
    the additive -inf mask on the same path, with the grid capped so every CTA
    walks several rows through its stage ring."""
    w = workloads.Workload("b_c", 1, 1, 12345, "f32", 8.0, 0.125, "none", False, False, 66, rows_override=40)
    x = workloads.make_inputs(w, device="cuda")["x"]
    mb = _mask((40, 12345), 0.1, 67)
    with H.grid_limit(3):
        y, taken = _run("auto", lambda: H.raw_forward_bool(x, mb, 0, 0, 1, w))
        y_add, taken_add = _run("auto", lambda: H.raw_forward(dict(x=x, mask=_additive(mb, torch.float32),
                                                                   mask_stride_b=0, mask_stride_h=0, heads=1), w))
    assert taken == taken_add == sms.SMS_PATH_CTA
    assert torch.equal(y, y_add)
    H.check_forward(H.to_np64(y), oracle.forward(x.cpu(), 12345, w.scale, False, mb.cpu()), torch.float32,
                    "bool fp32 S=12345 cta")


def test_bool_mask_autograd_and_in_place():
    B, Hh, S = 2, 4, 300
    g = torch.Generator(device="cuda").manual_seed(67)
    for dt in (torch.float32, torch.float16, torch.bfloat16):
        x = (torch.randn(B, Hh, S, S, generator=g, device="cuda") * 8).to(dt).requires_grad_(True)
        mb = _mask((B, 1, S, S), 0.2, 68)
        y = sms.scaled_mask_softmax(x, mb, 0.125, True)
        dy = torch.randn(B, Hh, S, S, generator=g, device="cuda").to(dt)
        y.backward(dy)
        torch.cuda.synchronize()
        y_add = sms.forward(x.detach(), _additive(mb, dt), 0.125, True)
        assert torch.equal(y.detach(), y_add)
        y_ref = oracle.forward(x.detach().cpu(), S, 0.125, True, mb.cpu(), S * S, 0, Hh)
        H.check_forward(H.to_np64(y).reshape(-1, S), y_ref.reshape(-1, S), dt, f"autograd bool {dt}")
        H.check_backward(H.to_np64(x.grad).reshape(-1, S), y.detach().cpu().reshape(-1, S),
                         dy.cpu().reshape(-1, S), 0.125, dt, f"autograd bool bwd {dt}")
        xi = x.detach().clone()
        sms.forward(xi, mb, 0.125, True, out=xi)  # y == x
        torch.cuda.synchronize()
        assert torch.equal(xi, y.detach())


@pytest.mark.parametrize("name", ["keypad_causal_bf16_s4096", "sweep_f16_s4099", "sweep_f32_s1024",
                                  "sweep_f32_s4099", "sweep_f32_s16384"])
def test_full_size_bool_mask(name):
    """Full-size workloads whose masks are 0 / -inf, with the mask given as
    bytes: every row against the oracle's boolean-mask path, and bit-equal to
    the additive-mask run when both take the same kernel family."""
    w = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(w, device="cuda")
    mb = torch.isinf(inp["mask"])
    y = H.raw_forward_bool(inp["x"], mb, inp["mask_stride_b"], inp["mask_stride_h"], inp["heads"], w)
    path_bool = sms.sms_last_path()
    torch.cuda.synchronize()
    assert sms.sms_device_error(torch.cuda.current_stream().cuda_stream) == 0
    H.check_all_rows(w, inp, y, None, name + " bool", bool_mask=mb)
    y_add = H.raw_forward(inp, w)
    path_add = sms.sms_last_path()
    torch.cuda.synchronize()
    if path_bool == path_add:
        assert torch.equal(y, y_add)
    else:
        H.check_all_rows(w, inp, y_add, None, name + " additive")
    del inp, y, y_add, mb
    torch.cuda.empty_cache()
