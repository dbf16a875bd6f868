"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Every kernel family (warp, cta, online, and the dispatcher's choice) is run on
the same seeded inputs as the oracle and compared element by element within
the stated tolerances (fp32 2e-6, fp16 1e-3, bf16 8e-3 absolute; masked
positions exactly 0; fp32 backward relative 1e-5).  Sizes span several CTAs,
ring wrap-arounds of the staged path and ragged tails; the full-size
workloads are checked on every row (the oracle over row chunks on the host)
plus properties that hold at any size.
"""
import dataclasses
import math

import numpy as np
import pytest
import torch

import oracle
import scaled_masked_softmax_gb300 as sms
from scaled_masked_softmax_gb300 import workloads
from tests import helpers as H

pytestmark = pytest.mark.gpu

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
WIDTHS = [1, 2, 3, 5, 8, 13, 16, 31, 33, 64, 100, 127, 128, 129, 255, 256, 500, 512, 513, 1000, 1023, 1024,
          1025, 1500, 1700, 1750, 2047, 2048, 2049, 3000, 3333, 3500, 4096, 4099, 5000, 8192, 12345, 16384, 20000,
          32768, 40000]
ROWS_FOR_PATH = {"auto": 300, "warp": 37, "stream": 2500, "ring": 3000, "cta": 1000, "online": 301}


def _wl(S, dt, rows, mask="SS", causal=False, B=1, Hh=1, seed=7, values="normal", fill=-math.inf):
    return workloads.Workload(f"t_{S}_{dt}", B, Hh, S, dt, 8.0, 0.125, mask, causal, True, seed,
                              pad_fill=fill, drop_p=0.15, rows_override=rows, mask_values=values)


def _budget_rows(S, rows):
    # keep every oracle call to a few million elements
    return max(3, min(rows, 12_000_000 // S))


def _run_fwd(w, inp, path):
    with H.forced_path(path):
        try:
            y = H.raw_forward(inp, w)
        except sms.SmsError as e:
            if e.status == 2:  # SMS_ERR_UNSUPPORTED: the forced path cannot take this width
                pytest.skip(f"{path} path does not take cols={w.cols}")
            raise
        taken = sms.sms_last_path()
    torch.cuda.synchronize()
    assert sms.sms_device_error(torch.cuda.current_stream().cuda_stream) == 0
    if path != "auto":
        assert taken == H.PATHS[path]
    return y


@pytest.mark.parametrize("path", ["auto", "warp", "stream", "ring", "cta", "online"])
@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("S", WIDTHS)
def test_forward_widths(S, dt, path):
    rows = _budget_rows(S, ROWS_FOR_PATH[path])
    w = _wl(S, dt, rows, causal=(WIDTHS.index(S) % 2 == 1))
    inp = H.make(w)
    y = _run_fwd(w, inp, path)
    H.check_forward(H.to_np64(y), H.oracle_forward(inp, w), DTYPES[dt], f"{path} S={S} {dt} causal={w.is_causal}")


@pytest.mark.parametrize("path", ["auto", "warp", "stream", "ring", "cta", "online"])
@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("kind", ["none", "SS", "B1SS", "BHSS"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S", [7, 100, 1000])
def test_forward_mask_layouts(S, causal, kind, dt, path):
    B, Hh = 2, 3
    fill = -10000.0 if kind == "B1SS" else -math.inf
    w = _wl(S, dt, None, mask=kind, causal=causal, B=B, Hh=Hh, seed=11, values="zero" if kind == "B1SS" else "normal",
            fill=fill)
    w = dataclasses.replace(w, pad_lo=0.3)
    inp = H.make(w)
    y = _run_fwd(w, inp, path)
    H.check_forward(H.to_np64(y), H.oracle_forward(inp, w), DTYPES[dt], f"{path} {kind} causal={causal} S={S} {dt}")


@pytest.mark.parametrize("path", ["auto", "warp", "stream", "ring", "cta", "online"])
@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("S", [1, 3, 31, 64, 129, 1000, 1024, 1025, 1700, 1750, 2048, 2049, 3333, 3500, 4099, 8192,
                               16384, 20000])
def test_backward_widths(S, dt, path):
    rows = _budget_rows(S, ROWS_FOR_PATH[path])
    causal = S % 2 == 1 or S in (1024, 8192)
    w = _wl(S, dt, rows, causal=causal)
    inp = H.make(w)
    y = H.raw_forward(inp, w)  # the stored y that the backward consumes
    with H.forced_path(path):
        try:
            dx = H.raw_backward(y, inp["dy"], w, causal_hint=False)
            dx_hint = H.raw_backward(y, inp["dy"], w, causal_hint=causal)
        except sms.SmsError as e:
            if e.status == 2:
                pytest.skip(f"{path} path does not take cols={S}")
            raise
    torch.cuda.synchronize()
    assert sms.sms_device_error(torch.cuda.current_stream().cuda_stream) == 0
    # the causal hint only skips reads of positions where y == 0: both results
    # meet the bound, and every position with y == 0 is +0 in both
    H.check_backward(H.to_np64(dx), y.cpu(), inp["dy"].cpu(), w.scale, DTYPES[dt], f"{path} bwd S={S} {dt}")
    H.check_backward(H.to_np64(dx_hint), y.cpu(), inp["dy"].cpu(), w.scale, DTYPES[dt], f"{path} bwd+hint S={S} {dt}")
    zero = y == 0
    assert torch.equal(dx[zero], torch.zeros_like(dx[zero]))
    assert torch.equal(dx_hint[zero], torch.zeros_like(dx_hint[zero]))
    assert not torch.signbit(dx_hint[zero]).any() and not torch.signbit(dx[zero]).any()


@pytest.mark.parametrize("name", ["tiny_causal_f32", "keypad_f32_s1024", "causal_spike_f16_s2048",
                                  "keypad_causal_bf16_s4096"])
def test_workload_scaled_forward_backward(name):
    base = workloads.WORKLOADS[name]
    w = workloads.scaled(base, B=min(base.B, 2), H=2) if name != "tiny_causal_f32" else base
    inp = workloads.make_inputs(w, device="cuda", with_dy=True)
    y = H.raw_forward(inp, w)
    torch.cuda.synchronize()
    y_ref = H.oracle_forward(inp, w)
    H.check_forward(H.to_np64(y), y_ref, w.torch_dtype, name)
    dx = H.raw_backward(y, inp["dy"], w, causal_hint=w.is_causal)
    torch.cuda.synchronize()
    H.check_backward(H.to_np64(dx), y.cpu(), inp["dy"].cpu(), w.scale, w.torch_dtype, name + " bwd")
    # end to end: the GPU backward on the GPU y against the oracle's fp64 chain
    dx_e2e = oracle.backward(y_ref, inp["dy"].cpu(), w.cols, w.scale)
    tol = {torch.float32: 1e-5, torch.float16: 2e-2, torch.bfloat16: 6e-2}[w.torch_dtype]
    rel = float(np.abs(H.to_np64(dx) - dx_e2e).max()) / max(float(np.abs(dx_e2e).max()), 1e-30)
    assert rel <= tol, f"{name}: end-to-end backward relative error {rel:.3e}"


@pytest.mark.parametrize("path", ["stream", "ring", "cta", "online"])
@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("S,kind,causal", [(8, "BHSS", True), (100, "B1SS", True), (1000, "SS", False),
                                           (2049, "B1SS", True), (4099, "SS", True)])
def test_persistent_kernels_walk_many_rows(S, kind, causal, dt, path):
    """Three CTAs only: every persistent CTA walks many rows (rings wrap,
    row cursors step across heads and batches)."""
    B, Hh = 3, 2
    rows = min(B * Hh * S, 6000 if S < 1000 else 900)
    fill = -10000.0 if kind == "B1SS" else -math.inf
    w = _wl(S, dt, rows, mask=kind, causal=causal, B=B, Hh=Hh, seed=23, values="zero" if kind == "B1SS" else "normal",
            fill=fill)
    inp = H.make(w)
    with H.grid_limit(3):
        y = _run_fwd(w, inp, path)
        with H.forced_path(path):
            dx = H.raw_backward(y, inp["dy"], w, causal_hint=causal)
        torch.cuda.synchronize()
    assert sms.sms_device_error(torch.cuda.current_stream().cuda_stream) == 0
    H.check_forward(H.to_np64(y), H.oracle_forward(inp, w), DTYPES[dt], f"{path} grid=3 S={S} {kind} {dt}")
    H.check_backward(H.to_np64(dx), y.cpu(), inp["dy"].cpu(), w.scale, DTYPES[dt], f"{path} grid=3 bwd S={S} {dt}")


LEN_WIDTHS = [1, 3, 8, 33, 100, 128, 129, 1000, 1024, 2049, 4099, 8192, 12345, 20000]


@pytest.mark.parametrize("path", ["auto", "warp", "stream", "ring", "cta", "online"])
@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("S", LEN_WIDTHS)
def test_key_lengths(S, dt, path):
    """sms_forward_lengths / sms_backward_lengths on every family: the oracle
    with key lengths, bit-identical to the same family run with the expanded
    [B,1,S,S] mask (0 below L_b, -inf from L_b on), lengths 0 (all-zero rows),
    1, beyond S and negative (clamped)."""
    causal = LEN_WIDTHS.index(S) % 2 == 0
    Hh = 2
    lengths = torch.tensor([S // 3 + 1, 0, 1, S, S + 5, -2], dtype=torch.int32)
    B = lengths.numel()
    rows = min(B * Hh * S, max(3, 12_000_000 // S))
    w = _wl(S, dt, rows, mask="none", causal=causal, B=B, Hh=Hh, seed=43)
    inp = H.make(w)
    L = lengths.cuda()
    # the same padding as an additive mask holding only the query rows the
    # rows reach: [batches, qmax, S], batch stride qmax*S
    nb, qmax = (rows + Hh * S - 1) // (Hh * S), min(S, rows)
    mask = torch.zeros(nb, qmax, S, device="cuda")
    for b in range(nb):
        mask[b, :, max(0, min(S, int(lengths[b]))):] = -math.inf
    mask = mask.to(DTYPES[dt])
    minp = dict(inp, mask=mask, mask_stride_b=qmax * S, mask_stride_h=0, heads=Hh)
    with H.forced_path(path):
        try:
            y = H.raw_forward_lengths(inp["x"], L, Hh, w)
            y_mask = H.raw_forward(minp, w)
            dx = H.raw_backward_lengths(y, inp["dy"], L, Hh, w, causal_hint=causal)
            dx_plain = H.raw_backward(y, inp["dy"], w, causal_hint=False)
        except sms.SmsError as e:
            if e.status == 2:
                pytest.skip(f"{path} path does not take cols={S}")
            raise
    torch.cuda.synchronize()
    assert sms.sms_device_error(torch.cuda.current_stream().cuda_stream) == 0
    assert torch.equal(y, y_mask), f"{path} S={S} {dt}: key lengths differ from the expanded mask"
    y_ref = oracle.forward(inp["x"].cpu(), S, w.scale, causal, heads=Hh, key_lengths=lengths)
    H.check_forward(H.to_np64(y), y_ref, DTYPES[dt], f"{path} lengths S={S} {dt} causal={causal}")
    H.check_backward(H.to_np64(dx), y.cpu(), inp["dy"].cpu(), w.scale, DTYPES[dt], f"{path} bwd lengths S={S} {dt}")
    H.check_backward(H.to_np64(dx_plain), y.cpu(), inp["dy"].cpu(), w.scale, DTYPES[dt], f"{path} bwd S={S} {dt}")
    zero = y == 0
    assert torch.equal(dx[zero], torch.zeros_like(dx[zero])) and not torch.signbit(dx[zero]).any()


@pytest.mark.parametrize("name", ["keypad_f32_s1024", "keypad_causal_bf16_s4096"])
def test_full_size_key_lengths(name):
    """The key-padding workloads at full size through the key-length entry
    points: sampled rows against the oracle, and equal to the additive-mask
    path on those rows."""
    w = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(w, device="cuda", with_dy=True)
    L = inp["key_lengths"]
    y = H.raw_forward_lengths(inp["x"], L, w.H, w)
    torch.cuda.synchronize()
    assert sms.sms_device_error(torch.cuda.current_stream().cuda_stream) == 0
    _properties(y, inp, w)
    y_mask = H.raw_forward(inp, w)
    torch.cuda.synchronize()
    # the same padding as the mask's -inf (or -10000, whose exponential is 0) entries: equal bit for bit
    assert torch.equal(y, y_mask)
    del y_mask
    dx = H.raw_backward_lengths(y, inp["dy"], L, w.H, w, causal_hint=w.is_causal)
    torch.cuda.synchronize()
    assert sms.sms_device_error(torch.cuda.current_stream().cuda_stream) == 0
    # every row, forward and backward, against the oracle
    H.check_all_rows(w, inp, y, dx, name + " lengths", key_lengths=L)
    del inp, y, dx
    torch.cuda.empty_cache()


def test_autograd_key_lengths():
    B, Hh, S = 3, 4, 200
    g = torch.Generator(device="cuda").manual_seed(47)
    for dt in (torch.float32, torch.float16, torch.bfloat16):
        x = (torch.randn(B, Hh, S, S, generator=g, device="cuda") * 8).to(dt).requires_grad_(True)
        L = torch.tensor([S, 73, 0], dtype=torch.int32, device="cuda")
        y = sms.scaled_mask_softmax(x, None, 0.125, True, key_lengths=L)
        dy = torch.randn(B, Hh, S, S, generator=g, device="cuda").to(dt)
        y.backward(dy)
        torch.cuda.synchronize()
        y_ref = oracle.forward(x.detach().cpu(), S, 0.125, True, heads=Hh, key_lengths=L.cpu())
        H.check_forward(H.to_np64(y).reshape(-1, S), y_ref.reshape(-1, S), dt, f"autograd lengths {dt}")
        H.check_backward(H.to_np64(x.grad).reshape(-1, S), y.detach().cpu().reshape(-1, S),
                         dy.cpu().reshape(-1, S), 0.125, dt, f"autograd lengths bwd {dt}")
        assert torch.all(y[2] == 0) and torch.all(x.grad[2] == 0)


@pytest.mark.parametrize("case", ["tiny_causal_f32", "f16_s1000_B1SS", "bf16_s4096_lengths", "f32_s20000_online",
                                  "f16_s2048_causal_ring"])
def test_cuda_graph_capture_and_replay(case):
    """Forward + backward captured into a CUDA graph after one eager call per
    shape (which does each kernel's one-time set-up), replayed on new inputs
    copied into the captured buffers: bit-identical to eager calls on those
    inputs.  Launch counts advance at capture, not at replay."""
    if case == "tiny_causal_f32":
        w = workloads.WORKLOADS["tiny_causal_f32"]
    elif case == "f16_s1000_B1SS":
        w = _wl(1000, "f16", None, mask="B1SS", B=2, Hh=3, seed=53, values="zero", fill=-10000.0)
    elif case == "bf16_s4096_lengths":
        w = workloads.scaled(workloads.WORKLOADS["keypad_causal_bf16_s4096"], B=2, H=2)
    elif case == "f32_s20000_online":
        w = _wl(20000, "f32", 300, causal=True, seed=59)
    else:
        w = workloads.scaled(workloads.WORKLOADS["causal_spike_f16_s2048"], B=1, H=2)
    use_len = case.endswith("lengths")
    a = workloads.make_inputs(w, device="cuda", with_dy=True)
    b = workloads.make_inputs(dataclasses.replace(w, seed=w.seed + 100), device="cuda", with_dy=True)

    def run(inp, y, dx):
        if use_len:
            H.raw_forward_lengths(inp["x"], inp["key_lengths"], w.H, w, y=y)
            H.raw_backward_lengths(y, inp["dy"], inp["key_lengths"], w.H, w, causal_hint=w.is_causal, dx=dx)
        else:
            H.raw_forward(inp, w, y=y)
            H.raw_backward(y, inp["dy"], w, causal_hint=w.is_causal, dx=dx)

    # eager references on both input sets
    y_a, dx_a = torch.empty_like(a["x"]), torch.empty_like(a["x"])
    y_b, dx_b = torch.empty_like(a["x"]), torch.empty_like(a["x"])
    run(a, y_a, dx_a)
    run(b, y_b, dx_b)
    torch.cuda.synchronize()
    # static buffers, captured on a side stream
    static = {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in a.items()}
    y_s, dx_s = torch.empty_like(a["x"]), torch.empty_like(a["x"])
    g = torch.cuda.CUDAGraph()
    n0 = sms.sms_launch_count()
    with torch.cuda.graph(g):
        run(static, y_s, dx_s)
    n_cap = sms.sms_launch_count() - n0
    assert n_cap == 2
    for src, y_ref, dx_ref in ((b, y_b, dx_b), (a, y_a, dx_a), (b, y_b, dx_b)):
        for k in ("x", "dy", "mask", "key_lengths"):
            if isinstance(static[k], torch.Tensor):
                static[k].copy_(src[k])
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y_s, y_ref) and torch.equal(dx_s, dx_ref)
    assert sms.sms_launch_count() - n0 == 2  # replays launch no new calls through the library
    assert sms.sms_device_error(torch.cuda.current_stream().cuda_stream) == 0


def test_spike_rows_are_one_hot():
    w = workloads.scaled(workloads.WORKLOADS["causal_spike_f16_s2048"], B=1, H=2)
    inp = workloads.make_inputs(w, device="cuda")
    y = H.raw_forward(inp, w)
    spikes = (inp["x"] == 60000).nonzero()
    assert spikes.shape[0] > 0
    for r, c in spikes.tolist():
        row = y[r]
        assert row[c].item() == 1.0
        assert int((row != 0).sum().item()) == 1


def test_fully_masked_rows_give_zero():
    for dt in ("f32", "f16", "bf16"):
        for S in (5, 64, 1000, 4099, 40000):
            w = _wl(S, dt, 4, mask="SS", values="zero")
            inp = H.make(w)
            inp["mask"][1, :] = -math.inf  # row 1 reads mask row 1: every key masked
            for path in ("auto", "warp", "stream", "ring", "cta", "online"):
                with H.forced_path(path):
                    try:
                        y = H.raw_forward(inp, w)
                        dx = H.raw_backward(y, inp["dy"], w, causal_hint=False)
                    except sms.SmsError as e:
                        if e.status == 2:  # the forced family cannot take this width
                            continue
                        raise
                torch.cuda.synchronize()
                assert torch.all(y[1] == 0) and torch.all(torch.isfinite(y))
                assert torch.all(dx[1] == 0) and torch.all(torch.isfinite(dx))


@pytest.mark.parametrize("path", ["warp", "stream", "ring", "cta", "online"])
def test_in_place(path):
    for dt, S in (("f32", 1000), ("bf16", 4099), ("f16", 1024)):
        w = _wl(S, dt, 257, causal=True)
        inp = H.make(w)
        with H.forced_path(path):
            try:
                y_ref = H.raw_forward(inp, w)
                x2 = inp["x"].clone()
                H.raw_forward(dict(inp, x=x2), w, y=x2)  # y is x
                dx_ref = H.raw_backward(y_ref, inp["dy"], w, causal_hint=True)
                dy2 = inp["dy"].clone()
                H.raw_backward(y_ref, dy2, w, causal_hint=True, dx=dy2)  # dx is dy
            except sms.SmsError as e:
                if e.status == 2:
                    continue
                raise
        torch.cuda.synchronize()
        assert torch.equal(x2, y_ref)
        assert torch.equal(dy2, dx_ref)


def test_rows_zero_and_one():
    w = _wl(64, "f32", 1, causal=False)
    inp = H.make(w)
    y = H.raw_forward(inp, w)
    torch.cuda.synchronize()
    H.check_forward(H.to_np64(y), H.oracle_forward(inp, w), torch.float32, "rows=1")
    n0 = sms.sms_launch_count()
    w0 = dataclasses.replace(w, rows_override=0)
    H.raw_forward(dict(inp, x=inp["x"][:0]), w0)
    assert sms.sms_launch_count() == n0


def test_autograd_functional_api():
    B, Hh, S = 2, 4, 128
    g = torch.Generator(device="cuda").manual_seed(3)
    for dt in (torch.float32, torch.float16, torch.bfloat16):
        x = (torch.randn(B, Hh, S, S, generator=g, device="cuda") * 8).to(dt).requires_grad_(True)
        L = torch.randint(S // 2, S + 1, (B,))
        m = torch.zeros(B, 1, S, S, device="cuda")
        for b in range(B):
            m[b, :, :, L[b]:] = -math.inf
        m = m.to(dt)
        y = sms.scaled_mask_softmax(x, m, 0.125, True)
        dy = torch.randn(B, Hh, S, S, generator=g, device="cuda").to(dt)
        y.backward(dy)
        torch.cuda.synchronize()
        y_ref = oracle.forward(x.detach().cpu(), S, 0.125, True, m.cpu(), S * S, 0, Hh)
        H.check_forward(H.to_np64(y).reshape(-1, S), y_ref.reshape(-1, S), dt, f"autograd {dt}")
        H.check_backward(H.to_np64(x.grad).reshape(-1, S), y.detach().cpu().reshape(-1, S),
                         dy.cpu().reshape(-1, S), 0.125, dt, f"autograd bwd {dt}")


def test_noncontiguous_and_misaligned_inputs():
    g = torch.Generator(device="cuda").manual_seed(5)
    x = torch.randn(2, 3, 64, 64, generator=g, device="cuda")
    xt = x.transpose(-1, -2)  # non-contiguous view
    y = sms.forward(xt, None, 0.5, True)
    y2 = sms.forward(xt.contiguous(), None, 0.5, True)
    assert torch.equal(y, y2)
    buf = torch.randn(64 * 64 + 1, generator=g, device="cuda")
    xm = buf[1:].view(64, 64)  # starts 4 bytes past a 16-byte boundary
    assert xm.data_ptr() % 16 != 0
    ym = sms.forward(xm, None, 0.5, False)
    torch.cuda.synchronize()
    H.check_forward(H.to_np64(ym), oracle.forward(xm.cpu(), 64, 0.5), torch.float32, "misaligned view")


def test_cpu_tensors_are_rejected():
    with pytest.raises(ValueError):
        sms.forward(torch.zeros(4, 4), None, 1.0, False)


# ---------------------------------------------------- full-size workloads ---

def _properties(y, inp, w):
    """Properties at any size: finite, rows sum to 1 (or 0 when fully masked),
    causal positions exactly 0."""
    assert bool(torch.isfinite(y).all())
    s = torch.sum(y, -1, dtype=torch.float32)
    tol = {torch.float32: 1e-5, torch.float16: 2e-3, torch.bfloat16: 1.6e-2}[y.dtype]
    assert float((s - 1).abs().max()) <= tol
    if w.is_causal:
        chunk = 4096
        cols = torch.arange(w.cols, device=y.device)
        for r0 in range(0, w.rows, chunk):
            r = torch.arange(r0, min(w.rows, r0 + chunk), device=y.device)
            above = cols[None, :] > (r % w.cols)[:, None]
            assert int(y[r0:r0 + r.numel()][above].ne(0).sum()) == 0


FULL = ["tiny_causal_f32", "keypad_f32_s1024", "causal_spike_f16_s2048", "keypad_causal_bf16_s4096"] + \
    [f"sweep_{dt}_s{S}" for dt in ("f16", "f32") for S in (128, 256, 512, 1000, 1024, 2048, 4099, 8192, 16384)]


@pytest.mark.parametrize("name", FULL)
def test_full_size_workload(name):
    w = workloads.WORKLOADS[name]
    with_dy = True
    inp = workloads.make_inputs(w, device="cuda", with_dy=with_dy)
    y = H.raw_forward(inp, w)  # dispatcher's choice, as the benchmark runs it
    torch.cuda.synchronize()
    assert sms.sms_device_error(torch.cuda.current_stream().cuda_stream) == 0
    _properties(y, inp, w)
    dx = H.raw_backward(y, inp["dy"], w, causal_hint=w.is_causal)
    torch.cuda.synchronize()
    assert sms.sms_device_error(torch.cuda.current_stream().cuda_stream) == 0
    # every row, forward and backward, against the oracle (in row chunks)
    chk = H.check_all_rows(w, inp, y, dx, name)
    assert chk.rows == w.rows
    del inp, y, dx
    torch.cuda.empty_cache()


@pytest.mark.parametrize("direction", ["forward", "backward"])
def test_ring_wait_that_runs_out_reports_and_recovers(direction):
    """The bounded-wait abort path, run on the GPU without a fault: with the
    test control on, each ring group's first wait is on a barrier nothing
    arrives at (bounded at 0.2 ms).  The kernel records SMS_DEVERR_RING_WAIT,
    drains its own bulk copies and returns; the error word reads once and
    clears, and the next call (control off) is correct."""
    w = _wl(2048, "f16", 900, mask="none", causal=True, seed=29)
    inp = H.make(w)
    st = torch.cuda.current_stream().cuda_stream
    y_ok = None
    if direction == "backward":
        with H.forced_path("ring"):
            y_ok = H.raw_forward(inp, w)
        torch.cuda.synchronize()
    prev = sms.sms_set_test_stall(200_000)
    try:
        with H.forced_path("ring"):
            if direction == "forward":
                H.raw_forward(inp, w)
            else:
                H.raw_backward(y_ok, inp["dy"], w, causal_hint=True)
        torch.cuda.synchronize()
        assert sms.sms_device_error(st) == 3  # SMS_DEVERR_RING_WAIT
    finally:
        sms.sms_set_test_stall(prev)
    assert sms.sms_device_error(st) == 0  # read once, then clear
    with H.forced_path("ring"):
        if direction == "forward":
            y = H.raw_forward(inp, w)
            torch.cuda.synchronize()
            H.check_forward(H.to_np64(y), H.oracle_forward(inp, w), torch.float16, "ring after a stall")
        else:
            dx = H.raw_backward(y_ok, inp["dy"], w, causal_hint=True)
            torch.cuda.synchronize()
            H.check_backward(H.to_np64(dx), y_ok.cpu(), inp["dy"].cpu(), w.scale, torch.float16, "ring bwd after a stall")
    assert sms.sms_device_error(st) == 0


@pytest.mark.parametrize("S,kind,rows_cut", [(4099, "B1SS", 77), (4100, "SS", 0), (4099, "SS", 1234)])
def test_mask_reuse_row_order(S, kind, rows_cut):
    """fp32 rows whose per-block mask is at least 64 MB go through the register
    row kernel in the mask-reuse order: every row still comes out once, right,
    with each batch's heads ([B,1,S,S]) or every head block ([S,S]) as the
    rows sharing a mask row, including a partial last batch or block."""
    B, Hh = 2, 3
    rows = B * Hh * S - rows_cut
    w = _wl(S, "f32", rows, mask=kind, B=B, Hh=Hh, seed=23)
    inp = H.make(w)
    y = _run_fwd(w, inp, "warp")
    chk = H.check_all_rows(w, inp, y, None, f"reuse order {kind} S={S} rows={rows}")
    assert chk.rows == rows
    del inp, y
    torch.cuda.empty_cache()
