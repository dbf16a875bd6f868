"""The attention backward for callers that cannot allocate device memory.

sms_attention_backward_static runs the same kernels as sms_attention_backward
but takes its scratch from a fixed array inside the library instead of a
workspace the caller allocates.  This file is collected last, so that a
failure here stops a run only after every other test has run; it passes on
its own in a fresh process and after the rest of the suite.

The check: two calls in a row through the C ABI (ctypes, no PyTorch
allocation between them), each on its own inputs, agree with the workspace
entry point on the same inputs within the bound the attention tests use.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention as A
from scaled_masked_softmax_gb300 import binding, workloads

pytestmark = pytest.mark.gpu

UNIT = {"f16": 2.0 ** -11, "bf16": 2.0 ** -8}
CODE = {"f16": binding.SMS_F16, "bf16": binding.SMS_BF16}


def _inputs(B, H, S, D, dt, seed, causal):
    q, k, v, d_o = workloads.attention_inputs(B, H, S, D, dt, seed=seed, device="cuda", with_do=True)
    o = torch.empty_like(q)
    lse = torch.empty(B, H, S, dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    scale = float(np.float32(1.0 / math.sqrt(D)))
    rc = binding.lib().sms_attention_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), None, 0, 0, 0, 0, o.data_ptr(),
                                             lse.data_ptr(), B, H, S, D, scale, int(causal), CODE[dt], st)
    assert rc == 0, binding.lib().sms_last_error()
    return q, k, v, o, lse, d_o, scale


def _grads(entry, q, k, v, o, lse, d_o, B, H, S, D, scale, causal, dt, ws=None):
    L = binding.lib()
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    st = torch.cuda.current_stream().cuda_stream
    common = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), d_o.data_ptr(), lse.data_ptr(), None, 0, 0, 0, 0,
              dq.data_ptr(), dk.data_ptr(), dv.data_ptr())
    if entry == "static":
        rc = L.sms_attention_backward_static(*common, B, H, S, D, scale, int(causal), CODE[dt], st)
    else:
        rc = L.sms_attention_backward(*common, ws.data_ptr(), ws.numel(), B, H, S, D, scale, int(causal), CODE[dt], st)
    assert rc == 0, L.sms_last_error()
    return dq, dk, dv


def _bound(q, k, v, d_o, scale, causal, dt):
    """The attention backward tests' bound, from the oracle's probabilities:
    6u M + u |X| + 1e-5 max M (+ the fp16 term), with M the first-order size
    of each gradient's terms."""
    qc, kc, vc, gc = q.cpu(), k.cpu(), v.cpu(), d_o.cpu()
    _, P = A.attention_forward(qc, kc, vc, scale, causal, return_probs=True)
    Q64, K64, V64, G64 = (np.abs(t.double().numpy()) for t in (qc, kc, vc, gc))
    Am = np.matmul(G64, np.swapaxes(V64, -1, -2))
    dlt = np.sum(P * Am, axis=-1, keepdims=True)
    G = P * (Am + dlt)
    mags = (abs(scale) * np.matmul(G, K64), abs(scale) * np.matmul(np.swapaxes(G, -1, -2), Q64),
            np.matmul(np.swapaxes(P, -1, -2), G64))
    u = UNIT[dt]
    extra = 0.0
    if dt == "f16":
        S = q.shape[2]
        extra = S * 2.0 ** -23 * (1 + abs(scale) * float((Am + dlt).max())) * max(Q64.max(), K64.max(), G64.max())
    return [6 * u * M + 1e-5 * float(M.max()) + extra + 1e-7 for M in mags]


@pytest.mark.parametrize("dt,causal", [("bf16", True), ("f16", False)])
def test_static_scratch_backward_twice_matches_the_workspace_entry_point(dt, causal):
    B, H, S, D = 2, 2, 300, 64
    ws_bytes = binding.lib().sms_attention_backward_workspace(B, H, S, D)
    assert 0 < ws_bytes <= binding.SMS_ATTN_STATIC_SCRATCH_BYTES
    for seed in (101, 202):  # two calls in a row, each on its own inputs
        q, k, v, o, lse, d_o, scale = _inputs(B, H, S, D, dt, seed, causal)
        got = _grads("static", q, k, v, o, lse, d_o, B, H, S, D, scale, causal, dt)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        ref = _grads("workspace", q, k, v, o, lse, d_o, B, H, S, D, scale, causal, dt, ws)
        torch.cuda.synchronize()
        assert binding.lib().sms_device_error(torch.cuda.current_stream().cuda_stream) == 0
        for name, a, b, bound in zip(("dQ", "dK", "dV"), got, ref, _bound(q, k, v, d_o, scale, causal, dt)):
            a64, b64 = a.double().cpu().numpy(), b.double().cpu().numpy()
            assert np.all(np.isfinite(a64)), f"{name}: non-finite"
            excess = np.abs(a64 - b64) - (bound + UNIT[dt] * np.abs(b64))
            assert float(excess.max()) <= 0, f"call {seed} {name}: differs by {float(np.abs(a64 - b64).max()):.3e}"


def test_static_scratch_rejects_problems_beyond_its_size():
    # a problem whose scratch exceeds the static array is refused with a clear error, before any launch
    L = binding.lib()
    S, D = 1 << 20, 128
    need = L.sms_attention_backward_workspace(1, 1, S, D)
    assert need > binding.SMS_ATTN_STATIC_SCRATCH_BYTES
    rc = L.sms_attention_backward_static(0x100000, 0x200000, 0x300000, 0x400000, 0x500000, 0x600000, None, 0, 0, 0, 0,
                                         0x700000, 0x800000, 0x900000, 1, 1, S, D, 0.1, 0, binding.SMS_BF16, None)
    assert rc == binding.SMS_ERR_INVALID_ARG
    assert "static" in L.sms_last_error().decode()
