"""The algorithmic bytes bench.py divides by (the roofline's numerator),
checked on small workloads by enumerating what each row reads and writes:
x at the kept positions (j <= q under causal), every distinct mask element
the rows touch (at the mask's element size: x's for an additive mask, one
byte for a boolean one), y / dx in full; y and dy at the kept positions in
the backward."""
import dataclasses
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from scaled_masked_softmax_gb300 import workloads  # noqa: E402


def _enumerate(w, inp, mask_eb):
    S, rows, eb = w.cols, w.rows, w.elem_bytes
    msb, msh, H = inp["mask_stride_b"], inp["mask_stride_h"], inp["heads"]
    x_read, mask_idx = 0, set()
    for r in range(rows):
        q, h, b = r % S, (r // S) % H, r // (S * H)
        kept = q + 1 if w.is_causal else S
        x_read += kept
        if inp["mask"] is not None:
            base = b * msb + h * msh + q * S
            mask_idx.update(range(base, base + kept))
    fwd = x_read * eb + len(mask_idx) * mask_eb + rows * S * eb
    bwd = 2 * x_read * eb + rows * S * eb
    return fwd, bwd


@pytest.mark.parametrize("name", ["tiny_causal_f32", "keypad_f32_s1024", "keypad_causal_bf16_s4096",
                                  "sweep_f16_s1000", "sweep_f32_s4099"])
@pytest.mark.parametrize("boolean", [False, True])
def test_algorithmic_bytes_match_enumeration(name, boolean):
    w = workloads.WORKLOADS[name]
    if w.rows_override is not None:  # [S,S] sweep: fewer rows than S, and more rows than S
        small = [dataclasses.replace(w, S=24, rows_override=17), dataclasses.replace(w, S=24, rows_override=61)]
    else:
        small = [workloads.scaled(w, B=2, H=3, S=20)]
    for ws in small:
        inp = workloads.make_inputs(ws, device="cpu", with_dy=False)
        if boolean and inp["mask"] is None:
            continue
        meb = 1 if boolean else None
        want_f, want_b = _enumerate(ws, inp, 1 if boolean else ws.elem_bytes)
        assert bench.fwd_bytes(ws, inp, False, meb) == want_f, ws
        assert bench.bwd_bytes(ws, inp) == want_b, ws


def test_cpu_baseline_reports_all_cores_and_one_thread():
    import oracle

    w = workloads.scaled(workloads.WORKLOADS["keypad_f32_s1024"], B=2, H=2, S=64)
    inp = workloads.make_inputs(w, device="cpu", with_dy=True)
    before = oracle.num_threads()
    r = bench.run_cpu_baseline(w, inp, 0.2)
    assert oracle.num_threads() == before  # the one-thread leg restores the thread count
    assert r["kind"] == "oracle" and r["cores"] == before and r["value"] > 0 and r["rows_per_s"] > 0
    assert r["single_thread"]["value"] > 0 and r["single_thread"]["rows_per_s"] > 0
    assert isinstance(r["cpu"], str) and r["cpu"]


@pytest.mark.parametrize("kind", ["none", "SS", "B1SS", "BHSS"])
@pytest.mark.parametrize("B,Hh,S,rows", [(3, 2, 8, None), (4, 3, 5, None), (1, 1, 7, 40), (2, 5, 4, None)])
@pytest.mark.parametrize("n_target", [1, 2, 3, 8, 100])
def test_e2e_blocks_keep_the_row_rule(kind, B, Hh, S, rows, n_target):
    """The pipelined end-to-end leg calls the kernels once per row block with
    shifted x / y / mask pointers: every row must land in exactly one block,
    and the block-relative row must reach the same query position and mask
    row as the absolute one."""
    if kind == "SS" and rows is None:
        rows = B * Hh * S
    w = workloads.Workload("t", B, Hh, S, "f32", 1.0, 1.0, kind, True, True, 1, rows_override=rows)
    msb, msh, H = w.mask_strides()
    blocks = bench.e2e_chunks(w, msb, msh, kind != "none", n_target)
    seen = []
    for r0, n, moff in blocks:
        assert n > 0
        for rr in range(n):
            r = r0 + rr
            seen.append(r)
            q, h, b = r % S, (r // S) % H, r // (S * H)
            q2, h2, b2 = rr % S, (rr // S) % H, rr // (S * H)
            assert q2 == q
            if kind != "none":
                assert moff + b2 * msb + h2 * msh + q2 * S == b * msb + h * msh + q * S
    assert seen == list(range(w.rows))
    assert len(blocks) <= max(1, n_target) or len(blocks) == -(-w.rows // (S * (H if kind in ("B1SS", "BHSS") else 1)))


def test_attention_flops_count_kept_pairs():
    # 2 S S D per product per head; causal keeps S (S + 1) / 2 pairs
    f, b = bench.attn_flops(2, 3, 8, 64, False)
    assert f == 2 * (2 * 8 * 8 * 64 * 6) and b == 5 * (2 * 8 * 8 * 64 * 6)
    fc, bc = bench.attn_flops(1, 1, 4, 16, True)
    pairs = sum(q + 1 for q in range(4))
    assert fc == 2 * 2 * pairs * 16 and bc == 5 * 2 * pairs * 16
