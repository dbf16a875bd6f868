"""Pins for the fp64 oracle against facts fixed outside the oracle itself.

Each check compares the oracle with something independent of it: closed forms
derived by hand (tests/golden/closed_forms.json), library routines on the cases
that reduce to them (numpy's fp16 and torch's bf16 widening, torch/scipy
softmax, torch autograd), invariants of softmax, and central finite
differences.  A dropped term, wrong sign, swapped index or misplaced stride in
oracle.c fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
DT = {"f64": torch.float64, "f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def _val(s):
    return float(eval(s, {"__builtins__": {}}, {"ln": math.log, "inf": math.inf}))


def _arr(rows, dtype):
    return torch.tensor([[_val(v) for v in row] for row in rows], dtype=torch.float64).to(dtype)


def _golden():
    with open(os.path.join(HERE, "golden", "closed_forms.json")) as f:
        return json.load(f)


# ---------------------------------------------------------------- fixtures ---

@pytest.mark.parametrize("case", _golden()["forward"], ids=lambda c: c["name"])
def test_forward_closed_forms(case):
    for dn in case["dtypes"]:
        dt = DT[dn]
        x = _arr(case["x"], dt)
        mask = _arr(case["mask"], dt) if "mask" in case else None
        if "bool_mask" in case:
            mask = torch.tensor(case["bool_mask"], dtype=torch.bool)
        scale = float(np.float32(_val(case["scale"])))
        y = oracle.forward(x, case["cols"], scale, case["is_causal"], mask,
                           case.get("mask_stride_b", 0), case.get("mask_stride_h", 0), case.get("heads", 1),
                           key_lengths=case.get("key_lengths"))
        want = _arr(case["y"], torch.float64).numpy()
        np.testing.assert_allclose(y, want, rtol=0, atol=1e-12, err_msg=f"{case['name']} {dn}")
        # masked entries are exactly zero, not merely small
        assert np.all(y[want == 0] == 0.0)


@pytest.mark.parametrize("case", _golden()["backward"], ids=lambda c: c["name"])
def test_backward_closed_forms(case):
    for dn in case["dtypes"]:
        dt = DT[dn]
        y = _arr(case["y"], dt)
        dy = _arr(case["dy"], dt)
        dx = oracle.backward(y, dy, case["cols"], _val(case["scale"]))
        want = _arr(case["dx"], torch.float64).numpy()
        np.testing.assert_allclose(dx, want, rtol=0, atol=1e-12, err_msg=f"{case['name']} {dn}")


# ---------------------------------------------------------------- decoders ---

def test_decode_f16_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = oracle.decode(bits, oracle.F16)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_decode_bf16_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.decode(bits, oracle.BF16)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_decode_one_element_equals_the_array_decoder():
    bits = np.arange(0, 65536, 97, dtype=np.uint32).astype(np.uint16)
    for code in (oracle.F16, oracle.BF16):
        whole = oracle.decode(bits, code)
        for i in range(0, bits.size, 7):
            one = oracle.decode_one(bits, i, code)
            assert (np.isnan(one) and np.isnan(whole[i])) or one == whole[i]


def test_decode_f32_random_bit_patterns():
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2**32, size=4096, dtype=np.uint64).astype(np.uint32)
    with np.errstate(invalid="ignore"):
        ref = bits.view(np.float32).astype(np.float64)
    got = oracle.decode(bits.view(np.float32))
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# ------------------------------------------------- library special cases ---

@pytest.mark.parametrize("dt", [torch.float64, torch.float32, torch.float16, torch.bfloat16])
@pytest.mark.parametrize("scale", [1.0, 0.125, 0.0883883476])
def test_forward_no_mask_matches_library_softmax(dt, scale):
    g = torch.Generator().manual_seed(11)
    x = (torch.randn(37, 53, generator=g, dtype=torch.float64) * 8).to(dt)
    s32 = float(np.float32(scale))
    y = oracle.forward(x, 53, s32)
    ref = torch.softmax(x.to(torch.float64) * s32, dim=-1).numpy()
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-13)
    import scipy.special

    np.testing.assert_allclose(y, scipy.special.softmax(x.to(torch.float64).numpy() * s32, axis=-1), rtol=0, atol=1e-13)


def _broadcast_case(B, H, S, dt, kind, causal, seed):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(B, H, S, S, generator=g, dtype=torch.float64) * 8).to(dt)
    shape = {"SS": (S, S), "B1SS": (B, 1, S, S), "BHSS": (B, H, S, S)}[kind]
    m = torch.randn(*shape, generator=g, dtype=torch.float64)
    drop = torch.rand(*shape, generator=g) < 0.2
    m = torch.where(drop, torch.tensor(-math.inf, dtype=torch.float64), m)
    m[..., 0] = 0.0  # keep column 0
    m = m.to(dt)
    strides = {"SS": (0, 0), "B1SS": (S * S, 0), "BHSS": (H * S * S, S * S)}[kind]
    return x, m, strides


@pytest.mark.parametrize("dt", [torch.float64, torch.float32, torch.float16, torch.bfloat16])
@pytest.mark.parametrize("kind", ["SS", "B1SS", "BHSS"])
@pytest.mark.parametrize("causal", [False, True])
def test_forward_masks_match_library_softmax(dt, kind, causal):
    B, H, S = 2, 3, 7
    x, m, (sb, sh) = _broadcast_case(B, H, S, dt, kind, causal, seed=5)
    scale = 0.125
    y = oracle.forward(x, S, scale, causal, m, sb, sh, H).reshape(B, H, S, S)
    s = x.to(torch.float64) * scale + m.to(torch.float64)  # torch broadcasting of [S,S] / [B,1,S,S]
    if causal:
        s = s + torch.triu(torch.full((S, S), -math.inf, dtype=torch.float64), diagonal=1)
    ref = torch.softmax(s, dim=-1).numpy()
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-13)


def test_row_index_selects_the_same_rows():
    B, H, S = 2, 3, 9
    x, m, (sb, sh) = _broadcast_case(B, H, S, torch.float32, "B1SS", True, seed=3)
    full = oracle.forward(x, S, 0.125, True, m, sb, sh, H).reshape(-1, S)
    idx = np.array([0, 5, 9, 26, 27, 40, 53], dtype=np.int64)
    xr = x.reshape(-1, S)[torch.from_numpy(idx)]
    part = oracle.forward(xr, S, 0.125, True, m, sb, sh, H, row_index=idx)
    np.testing.assert_array_equal(part, full[idx])


# -------------------------------------------------------------- invariants ---

def test_invariants_sum_zero_shift_uniform():
    g = torch.Generator().manual_seed(2)
    S = 33
    x = torch.randn(40, S, generator=g, dtype=torch.float64) * 8
    m = torch.where(torch.rand(S, S, generator=g) < 0.3, -math.inf, 0.0).to(torch.float64)
    m[:, 0] = 0
    xs = x[:S]
    y = oracle.forward(xs, S, 0.125, False, m)
    np.testing.assert_allclose(y.sum(-1), 1.0, rtol=0, atol=1e-14)
    assert np.all(y[np.isneginf(m.numpy())] == 0.0)
    # adding c/scale to every x of a row leaves y unchanged (8*c is exact here)
    for c in (1.0, -1.0, 100.0, -100.0):
        y2 = oracle.forward(xs + 8.0 * c, S, 0.125, False, m)
        np.testing.assert_allclose(y2, y, rtol=0, atol=1e-12)
    # a constant row gives 1/n_kept on kept positions
    yc = oracle.forward(torch.full((S, S), 3.5, dtype=torch.float64), S, 0.125, False, m)
    kept = np.isfinite(m.numpy())
    want = kept / kept.sum(-1, keepdims=True)
    np.testing.assert_allclose(yc, want, rtol=0, atol=1e-15)
    # causal rows of a constant tensor give 1/(q+1)
    yq = oracle.forward(torch.zeros(2 * S, S, dtype=torch.float64), S, 1.0, True)
    for r in range(2 * S):
        q = r % S
        np.testing.assert_allclose(yq[r, : q + 1], 1.0 / (q + 1), rtol=0, atol=1e-15)
        assert np.all(yq[r, q + 1:] == 0.0)


def test_permuting_columns_permutes_output():
    g = torch.Generator().manual_seed(4)
    S = 17
    x = torch.randn(S, S, generator=g, dtype=torch.float64) * 8
    m = torch.randn(S, S, generator=g, dtype=torch.float64)
    perm = torch.randperm(S, generator=g)
    y = oracle.forward(x, S, 0.5, False, m)
    yp = oracle.forward(x[:, perm], S, 0.5, False, m[:, perm])
    np.testing.assert_allclose(yp, y[:, perm.numpy()], rtol=0, atol=1e-15)


def test_two_element_logistic_closed_form():
    rng = np.random.default_rng(0)
    for _ in range(50):
        a, b = rng.normal(0, 10, 2)
        sc = float(np.float32(rng.uniform(0.05, 2)))
        y = oracle.forward(np.array([[a, b]]), 2, sc)
        want0 = 1.0 / (1.0 + math.exp((b - a) * sc))
        assert abs(y[0, 0] - want0) < 1e-14 and abs(y[0, 1] - (1 - want0)) < 1e-14


def test_scale_acts_on_x_only():
    g = torch.Generator().manual_seed(9)
    x = torch.randn(6, 10, generator=g, dtype=torch.float64)
    m = torch.randn(10, 10, generator=g, dtype=torch.float64)
    y = oracle.forward(x, 10, 3.0, False, m)
    y1 = oracle.forward(x * 3.0, 10, 1.0, False, m)
    np.testing.assert_allclose(y, y1, rtol=0, atol=1e-14)


def test_fully_masked_rows_are_zero_and_nan_free():
    S = 8
    m = torch.zeros(S, S, dtype=torch.float32)
    m[3, :] = -math.inf
    y = oracle.forward(torch.randn(S, S), S, 1.0, False, m)
    assert np.all(y[3] == 0.0)
    assert np.all(np.isfinite(y))


# ---------------------------------------------------------------- backward ---

def test_backward_matches_central_differences():
    g = torch.Generator().manual_seed(13)
    S, scale = 24, 0.37
    x = torch.randn(5, S, generator=g, dtype=torch.float64) * 3
    m = torch.randn(S, S, generator=g, dtype=torch.float64)
    m[:, 5] = -math.inf
    dy = torch.randn(5, S, generator=g, dtype=torch.float64)
    y = oracle.forward(x, S, scale, True, m)
    dx = oracle.backward(y, dy.numpy(), S, scale)
    h = 1e-6
    fd = np.zeros_like(dx)
    for i in range(5):
        for j in range(S):
            xp = x.clone(); xp[i, j] += h
            xm = x.clone(); xm[i, j] -= h
            lp = (oracle.forward(xp, S, scale, True, m) * dy.numpy()).sum()
            lm = (oracle.forward(xm, S, scale, True, m) * dy.numpy()).sum()
            fd[i, j] = (lp - lm) / (2 * h)
    assert np.max(np.abs(dx - fd)) <= 1e-6 * max(1.0, np.max(np.abs(fd)))


def test_backward_matches_autograd_and_jacobian():
    g = torch.Generator().manual_seed(21)
    S, scale = 19, 0.125
    x = (torch.randn(12, S, generator=g, dtype=torch.float64) * 8).requires_grad_(True)
    m = torch.where(torch.rand(12, S, generator=g) < 0.2, -math.inf, 0.0).to(torch.float64)
    m[:, 0] = 0
    dy = torch.randn(12, S, generator=g, dtype=torch.float64)
    yt = torch.softmax(x * scale + m, dim=-1)
    (gx,) = torch.autograd.grad(yt, x, dy)
    y = yt.detach().numpy()
    dx = oracle.backward(y, dy.numpy(), S, scale)
    np.testing.assert_allclose(dx, gx.numpy(), rtol=0, atol=1e-13)
    # explicit Jacobian of softmax: scale * (diag(y) - y y^T), symmetric
    for i in range(12):
        J = scale * (np.diag(y[i]) - np.outer(y[i], y[i]))
        np.testing.assert_allclose(dx[i], J.T @ dy[i].numpy(), rtol=0, atol=1e-13)
    np.testing.assert_allclose(dx.sum(-1), 0.0, rtol=0, atol=1e-13)
    # a constant upstream gradient gives no gradient at all
    dc = oracle.backward(y, np.full_like(y, 2.5), S, scale)
    np.testing.assert_allclose(dc, 0.0, rtol=0, atol=1e-15)


def test_backward_mixed_dtypes():
    g = torch.Generator().manual_seed(1)
    y = torch.softmax(torch.randn(4, 16, generator=g, dtype=torch.float64), -1)
    dy = torch.randn(4, 16, generator=g).to(torch.bfloat16)
    dx = oracle.backward(y, dy, 16, 0.5)
    want = oracle.backward(y, dy.to(torch.float64), 16, 0.5)
    np.testing.assert_array_equal(dx, want)


def test_oracle_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.forward(np.zeros((2, 3)), 4, 1.0)
    with pytest.raises(ValueError):
        oracle.backward(np.zeros((2, 3)), np.zeros((2, 4)), 3, 1.0)


# ------------------------------------------------------------ key lengths ---

@pytest.mark.parametrize("dt", [torch.float64, torch.float32, torch.float16, torch.bfloat16])
@pytest.mark.parametrize("causal", [False, True])
def test_key_lengths_equal_an_expanded_minus_inf_mask(dt, causal):
    """The key-length path and the additive-mask path of the oracle are two
    different mechanisms; a [B,1,S,S] mask of 0 below L_b and -inf from L_b
    on must give the same result bit for bit."""
    g = torch.Generator().manual_seed(31)
    B, H, S = 3, 2, 37
    x = (torch.randn(B * H * S, S, generator=g, dtype=torch.float64) * 8).to(dt)
    L = torch.tensor([0, 17, 37], dtype=torch.int32)
    mask = torch.zeros(B, 1, S, S, dtype=torch.float64)
    for b in range(B):
        mask[b, :, :, int(L[b]):] = -math.inf
    y_len = oracle.forward(x, S, 0.125, causal, heads=H, key_lengths=L)
    y_mask = oracle.forward(x, S, 0.125, causal, mask.to(dt), S * S, 0, H)
    assert np.array_equal(y_len, y_mask)


@pytest.mark.parametrize("dt", [torch.float64, torch.float32, torch.float16, torch.bfloat16])
def test_key_lengths_match_library_softmax(dt):
    """Rows with at least one kept key against torch.softmax of the scores
    with the padded keys filled with -inf."""
    g = torch.Generator().manual_seed(37)
    B, H, S = 4, 3, 50
    x = (torch.randn(B * H * S, S, generator=g, dtype=torch.float64) * 8).to(dt)
    L = torch.tensor([1, 25, 49, 50], dtype=torch.int32)
    y = oracle.forward(x, S, 0.125, False, heads=H, key_lengths=L)
    s = x.to(torch.float64) * float(np.float32(0.125))
    b = torch.arange(B * H * S) // (H * S)
    pad = torch.arange(S)[None, :] >= L.to(torch.int64)[b][:, None]
    ref = torch.softmax(s.masked_fill(pad, -math.inf), dim=-1).numpy()
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-14)
    assert np.all(y[pad.numpy()] == 0.0)


def test_key_lengths_with_row_index_and_clamping():
    """A row sample by row_index picks each row's batch; lengths below 0 or
    above cols are clamped."""
    g = torch.Generator().manual_seed(41)
    B, H, S = 3, 2, 9
    x = torch.randn(B * H * S, S, generator=g, dtype=torch.float64)
    L = torch.tensor([-5, 4, 100], dtype=torch.int32)
    full = oracle.forward(x, S, 1.0, True, heads=H, key_lengths=L)
    idx = np.array([53, 0, 20, 36, 17], dtype=np.int64)
    part = oracle.forward(x[torch.as_tensor(idx)], S, 1.0, True, heads=H, key_lengths=L, row_index=idx)
    assert np.array_equal(part, full[idx])
    assert np.all(full[: H * S] == 0.0)  # L = -5 -> 0: every key of batch 0 masked
    np.testing.assert_array_equal(full[2 * H * S:], oracle.forward(x[2 * H * S:], S, 1.0, True))  # L = 100 -> S


# ----------------------------------------------------------- boolean masks ---

@pytest.mark.parametrize("dt", [torch.float64, torch.float32, torch.float16, torch.bfloat16])
@pytest.mark.parametrize("kind", ["SS", "B1SS", "BHSS"])
@pytest.mark.parametrize("causal", [False, True])
def test_bool_mask_equals_additive_minus_inf_mask(dt, kind, causal):
    """The boolean-mask path and the additive-mask path of the oracle are two
    mechanisms; a boolean mask and the additive mask holding -inf where it is
    true (0 elsewhere) must give the same result bit for bit, on every
    broadcast layout."""
    g = torch.Generator().manual_seed(61)
    B, H, S = 2, 3, 29
    x = (torch.randn(B * H * S, S, generator=g, dtype=torch.float64) * 8).to(dt)
    shape = {"SS": (S, S), "B1SS": (B, 1, S, S), "BHSS": (B, H, S, S)}[kind]
    sb, sh = {"SS": (0, 0), "B1SS": (S * S, 0), "BHSS": (H * S * S, S * S)}[kind]
    bm = torch.rand(shape, generator=g) < 0.3
    bm[..., 0] = False
    bm.view(-1, S)[3] = True  # one fully masked mask row
    add = torch.zeros(shape, dtype=torch.float64).masked_fill(bm, -math.inf).to(dt)
    y_bool = oracle.forward(x, S, 0.125, causal, bm, sb, sh, H)
    y_add = oracle.forward(x, S, 0.125, causal, add, sb, sh, H)
    assert np.array_equal(y_bool, y_add)


def test_bool_mask_matches_library_softmax():
    """torch.softmax of the scores with the true positions filled with -inf
    (rows with at least one kept key), uint8 and bool masks alike."""
    g = torch.Generator().manual_seed(67)
    S = 40
    x = torch.randn(S, S, generator=g, dtype=torch.float64) * 8
    bm = torch.rand(S, S, generator=g) < 0.5
    bm[:, 7] = False
    ref = torch.softmax((x * float(np.float32(0.125))).masked_fill(bm, -math.inf), -1).numpy()
    for m in (bm, bm.to(torch.uint8) * 3):  # any nonzero byte masks
        y = oracle.forward(x, S, 0.125, False, m)
        np.testing.assert_allclose(y, ref, rtol=0, atol=1e-14)
        assert np.all(y[bm.numpy()] == 0.0)
