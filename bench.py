#!/usr/bin/env python3
"""Benchmark of the fused ScaledMaskSoftmax on GB300.

One step = one pass of the whole hot path over one batch: the forward
(load + scale + mask + causal, row max, exp + sum, normalise + store) and the
backward (row dot, gradient) through the C ABI, on inputs already resident in
HBM.  Default workload: [4,32,4096,4096] bf16 scores (d_k = 128, scale
1/sqrt(128)) with a [4,1,4096,4096] key-padding mask (-inf fill) and the causal
flag, forward then backward (with the causal hint) with dy ~ N(0,1).

Prints ONE JSON line (rank 0).  ``--impl reference`` times the fp64 CPU oracle
instead, on bounded samples of the same workload.  ``--all`` additionally
writes one JSON line per workload to the file given.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "fused masked-softmax fwd/bwd achieved HBM GB/s and % of GB300 peak; rows/s"
DEFAULT_WORKLOAD = "keypad_causal_bf16_s4096"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, nominal
DTYPE_NAME = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}


# ----------------------------------------------------------------- helpers ---

def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _kernel_hash() -> str:
    """Hash of the softmax kernel sources and their dispatcher (the attention
    kernels, sms_attn*, are not part of it)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "scaled_masked_softmax_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.startswith(("sms_attn", "sms_tc")):
            continue
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def _traffic_record(workload: str, kernel: str):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("kernel_hash") != _kernel_hash():
        return None
    rec = d.get("workloads", {}).get(workload, {}).get(kernel)
    if not rec:
        return None
    return rec.get("bytes_per_launch")


def _kept_elems(w, inp) -> float:
    """Elements a key-length run reads per tensor: min(L_b, q + 1 under causal) per row."""
    L = inp["key_lengths"].to("cpu", torch.float64).clamp(0, w.cols)
    r = torch.arange(w.rows, dtype=torch.float64)
    b = torch.div(r, w.H * w.cols, rounding_mode="floor").long()
    lim = L[b]
    if w.is_causal:
        lim = torch.minimum(lim, torch.remainder(r, w.cols) + 1)
    return float(lim.sum())


def fwd_bytes(w, inp, lengths=False, mask_eb=None) -> int:
    """Algorithmic bytes of one forward: x read (only j <= q under causal),
    unique mask bytes read (same causal rule; mask_eb bytes per mask element,
    1 for a boolean mask, else x's), y written in full.  With key lengths: x
    read only below min(L_b, q + 1), the lengths array, no mask."""
    eb = w.elem_bytes
    meb = eb if mask_eb is None else mask_eb
    rows, S = w.rows, w.cols
    if lengths:
        return int(_kept_elems(w, inp) * eb + inp["key_lengths"].numel() * 4 + rows * S * eb)
    if w.is_causal:
        # row q reads q+1 elements
        q = torch.arange(rows, dtype=torch.float64) % S
        x_read = float((q + 1).sum()) * eb
    else:
        x_read = rows * S * eb
    mask_read = 0.0
    if inp["mask"] is not None:
        if w.mask == "B1SS":
            nb = math.ceil(rows / (w.H * S))
            per_q = (torch.arange(S, dtype=torch.float64) + 1).sum() if w.is_causal else S * S
            mask_read = float(nb * per_q) * meb
        else:  # [S,S] (or full): rows touch min(rows, S) distinct mask rows per mask head
            nq = min(rows, S)
            per_q = float((torch.arange(nq, dtype=torch.float64) + 1).sum()) if w.is_causal else nq * S
            mask_read = per_q * meb
    return int(x_read + mask_read + rows * S * eb)


def bwd_bytes(w, inp=None, lengths=False) -> int:
    """Algorithmic bytes of one backward: y and dy read (only j <= q with the
    causal hint, only below L_b with key lengths), dx written in full."""
    eb = w.elem_bytes
    rows, S = w.rows, w.cols
    if lengths:
        return int(_kept_elems(w, inp) * 2 * eb + inp["key_lengths"].numel() * 4 + rows * S * eb)
    if w.is_causal:
        q = torch.arange(rows, dtype=torch.float64) % S
        read = float((q + 1).sum()) * 2 * eb
    else:
        read = rows * S * 2 * eb
    return int(read + rows * S * eb)


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.sel = []
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            self.sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            self.sel = []
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="sms_clocks_", suffix=".csv")
            self.f = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(["nvidia-smi"] + self.sel + [f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], None, set()
        with open(self.path) as f:
            lines = f.readlines()
        try:
            os.unlink(self.path)
        except OSError:
            pass
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                s, m = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            sm.append(s)
            mx = m
            for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"),
                               parts[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------- ranks (weak) ---

def dist_env():
    """(world, rank, local_rank) from the launcher's environment; one process
    per GPU, each running the whole workload on its own rows (replicas)."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init_dist(world, rank):
    if world > 1:
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend, rank=rank, world_size=world)


def max_over_ranks(ms, world, device=None):
    """The slowest rank's time: the job is done when every rank is."""
    if world <= 1:
        return ms
    on_gpu = torch.distributed.get_backend() == "nccl"
    t = torch.tensor([ms], dtype=torch.float64, device=device if on_gpu else "cpu")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(step_bytes, world, step_ms):
    """Whole-job throughput: every rank moves step_bytes per step (weak
    scaling), all of them within the slowest rank's step time."""
    return step_bytes * world / (step_ms * 1e6)


# ------------------------------------------------------------------ ours ---

def _workload(args):
    """The named workload, or (``--bh B,H``) the same distributions at another
    batch and head count (small profiling captures of the same kernels)."""
    from scaled_masked_softmax_gb300 import workloads

    w = workloads.WORKLOADS[args.workload]
    bh = getattr(args, "bh", None)
    if bh:
        b, h = (int(v) for v in bh.split(","))
        w = workloads.scaled(w, B=b, H=h)
    return w


def run_ours(args, rank, world, device):
    import scaled_masked_softmax_gb300 as sms
    from scaled_masked_softmax_gb300 import workloads

    w = _workload(args)
    torch.cuda.set_device(device)
    inp = workloads.make_inputs(w, device=device, with_dy=True)
    x, mask, dy = inp["x"], inp["mask"], inp["dy"]
    y = torch.empty_like(x)
    dx = torch.empty_like(x)
    stream = torch.cuda.current_stream(device)
    st = stream.cuda_stream
    dt = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}[x.dtype]
    mptr = None if mask is None else mask.data_ptr()
    mnum = 0 if mask is None else mask.numel()
    L = sms.binding.lib()

    use_len = bool(getattr(args, "lengths", False))
    if use_len and inp["key_lengths"] is None:
        raise RuntimeError(f"--lengths: workload {w.name} has no key-padding mask")
    lptr = inp["key_lengths"].data_ptr() if use_len else None
    use_bool = bool(getattr(args, "bool_mask", False))
    if use_bool:
        if mask is None or use_len:
            raise RuntimeError(f"--bool-mask: workload {w.name} has no mask tensor (or --lengths is set)")
        mbool = (mask != 0).contiguous()  # the workloads' masks hold 0 (kept) or -inf / -10000 (masked)
        mptr = mbool.data_ptr()

    def fwd():
        if use_bool:
            rc = L.sms_forward_bool(x.data_ptr(), mptr, mnum, inp["mask_stride_b"], inp["mask_stride_h"],
                                    inp["heads"], y.data_ptr(), w.rows, w.cols, w.scale, int(w.is_causal), dt, st)
        elif use_len:
            rc = L.sms_forward_lengths(x.data_ptr(), lptr, w.H, y.data_ptr(), w.rows, w.cols, w.scale,
                                       int(w.is_causal), dt, st)
        else:
            rc = L.sms_forward(x.data_ptr(), mptr, mnum, inp["mask_stride_b"], inp["mask_stride_h"], inp["heads"],
                               y.data_ptr(), w.rows, w.cols, w.scale, int(w.is_causal), dt, st)
        if rc:
            raise RuntimeError(sms.sms_last_error())

    def bwd():
        if use_len:
            rc = L.sms_backward_lengths(y.data_ptr(), dy.data_ptr(), dx.data_ptr(), lptr, w.H, w.rows, w.cols,
                                        w.scale, int(w.is_causal), dt, st)
        else:
            rc = L.sms_backward(y.data_ptr(), dy.data_ptr(), dx.data_ptr(), w.rows, w.cols, w.scale,
                                int(w.is_causal), dt, st)
        if rc:
            raise RuntimeError(sms.sms_last_error())

    fb, bb = fwd_bytes(w, inp, use_len, 1 if use_bool else None), bwd_bytes(w, inp, use_len)
    step_bytes = fb + bb
    working_set = (x.numel() * 4 * x.element_size()) + (0 if mask is None else mask.numel() * mask.element_size())
    flush = working_set < 2 * L2_BYTES
    scratch = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=device) if flush else None

    for _ in range(max(args.warmup, 3)):
        fwd()
        fp = sms.sms_last_path()
        bwd()
        bp = sms.sms_last_path()
    taken = (fp, bp)
    torch.cuda.synchronize(device)

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(device)
    if rank == 0:
        clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(device)
    n_launch0 = sms.sms_launch_count()
    t0.record(stream)
    for i in range(K):
        if flush:
            scratch.add_(1.0)  # evict the previous step's data from L2 (outside the per-kernel events)
        ev[i][0].record(stream)
        fwd()
        ev[i][1].record(stream)
        bwd()
        ev[i][2].record(stream)
    t1.record(stream)
    torch.cuda.synchronize(device)
    if world > 1:
        torch.distributed.barrier()
    n_launch = sms.sms_launch_count() - n_launch0
    clk = clocks.stop() if rank == 0 else None

    fwd_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    bwd_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(K)]
    region_ms = t0.elapsed_time(t1)
    kern_ms = sum(fwd_ms) + sum(bwd_ms)
    # with an L2 flush between steps the step time is the kernels' own time
    step_ms = (kern_ms if flush else region_ms) / K

    step_ms = max_over_ranks(step_ms, world, device)

    peak, peak_kind = _peaks()
    f_ms, b_ms = statistics.mean(fwd_ms), statistics.mean(bwd_ms)
    fwd_path, bwd_path = taken

    def _kernel(path, ms_list, nbytes):
        ms = statistics.mean(ms_list)  # the average launch duration (the roofline's denominator)
        return {"path": sms.PATH_NAMES[path], "ms": round(ms, 4), "median_ms": round(statistics.median(ms_list), 4),
                "alg_bytes": nbytes, "gbs": round(nbytes / ms / 1e6, 1), "frac_of_peak": round(nbytes / ms / 1e6 / peak, 4)}

    kernels = {"forward": _kernel(fwd_path, fwd_ms, fb), "backward": _kernel(bwd_path, bwd_ms, bb)}
    dom = "backward" if b_ms * K >= f_ms * K else "forward"
    wkey = w.name + ("+lengths" if use_len else "+bool" if use_bool else "")
    traffic = _traffic_record(wkey, dom)
    roof = {"kernel": dom, "bound": "hbm", "achieved": kernels[dom]["gbs"], "peak": peak, "unit": "GB/s",
            "frac": round(kernels[dom]["gbs"] / peak, 4), "traffic": traffic, "peak_source": peak_kind,
            "frac_of_nominal": round(kernels[dom]["gbs"] / NOMINAL_HBM_GBS, 4),
            # DRAM bytes the profiler counted per launch over the same event-timed launch duration
            "traffic_gbs": None if traffic is None else round(traffic / kernels[dom]["ms"] / 1e6, 1)}
    for name, k in kernels.items():
        t = _traffic_record(wkey, name)
        k["ncu_dram_bytes"] = t
        k["ncu_dram_gbs"] = None if t is None else round(t / k["ms"] / 1e6, 1)

    graph = None
    if getattr(args, "graph", 0) and args.graph > 0:
        # the same step replayed from a CUDA graph of `args.graph` steps (launch
        # overhead amortised; each kernel did its one-time set-up in the warm-up)
        n = args.graph
        gs = torch.cuda.Stream(device)
        gs.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(gs):
            st_saved = st
            st = gs.cuda_stream
            with torch.cuda.graph(g, stream=gs):
                for _ in range(n):
                    fwd()
                    bwd()
            st = st_saved
        stream.wait_stream(gs)
        reps = max(1, K // n)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize(device)
        ga, gb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ga.record(stream)
        for _ in range(reps):
            g.replay()
        gb.record(stream)
        torch.cuda.synchronize(device)
        g_ms = ga.elapsed_time(gb) / (reps * n)
        graph = {"steps_per_graph": n, "replays": reps, "ms_per_step": round(g_ms, 5),
                 "value": round(step_bytes / (g_ms * 1e6), 1), "unit": "GB/s",
                 "rows_per_s": round(w.rows / (g_ms / 1e3), 1),
                 "note": "fwd+bwd steps replayed from one CUDA graph on inputs resident in HBM"}

    value = aggregate_gbs(step_bytes, world, step_ms)
    res = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": DTYPE_NAME[x.dtype], "data": "synthetic (seeded, see workloads.py)",
        "config": {"workload": w.name, "shape": [w.B, w.H, w.S, w.S] if w.rows_override is None else [w.rows, w.S],
                   "rows": w.rows, "cols": w.cols,
                   "mask": ("key lengths int32 [B] (sms_forward_lengths)" if use_len else
                            f"{w.mask} as bytes (sms_forward_bool)" if use_bool else w.mask),
                   "is_causal": w.is_causal,
                   "step": "forward + backward (dy ~ N(0,1))", "scale": w.scale,
                   "l2": ("flushed between steps (2x L2 write), step = kernel time" if flush
                          else "inputs larger than L2, no flush"),
                   "parallelism": f"replicas x{world} (independent rows per GPU)"},
        "pct_of_peak": round(100 * value / world / peak, 2),
        "pct_of_peak_basis": f"{peak_kind} copy bandwidth {peak} GB/s",
        "pct_of_nominal": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "rows_per_s": round(w.rows * world / (step_ms / 1e3), 1),
        "kernels": kernels, "roofline": roof, "gpu_launches": int(n_launch), "graph": graph,
        "clocks": clk,
    }
    return res, (w, inp, y, dx)


def e2e_chunks(w, msb, msh, has_mask, n_target=8):
    """Row blocks of the pipelined end-to-end leg: (first row, rows, mask
    element offset).  A block starts where the kernels' row rule (q = r mod S,
    h, b from r) still holds for its block-relative rows: at a batch boundary
    when the mask varies by batch or head (the mask pointer then moves to that
    batch), else at a multiple of S rows (a shared or absent mask)."""
    per_batch = has_mask and (msb != 0 or msh != 0)
    unit = w.H * w.cols if per_batch else w.cols
    n_units = -(-w.rows // unit)
    per = max(1, -(-n_units // n_target))
    out = []
    for u0 in range(0, n_units, per):
        r0 = u0 * unit
        n = min(w.rows, (u0 + per) * unit) - r0
        moff = (r0 // (w.H * w.cols)) * msb if per_batch else 0
        out.append((r0, n, moff))
    return out


def run_e2e(args, w, inp, device, steps):
    """Same metric through the C ABI with host buffers.  Every step copies x,
    dy (and the mask) in from pinned host memory, runs the forward and the
    backward, and copies y and dx back out.  The rows are cut into blocks
    (``e2e_chunks``) on three streams: the copy-in of block i+1, the kernels
    of block i and the copy-out of block i-1 overlap, and the two copy
    directions run at once."""
    import scaled_masked_softmax_gb300 as sms

    L = sms.binding.lib()
    mask = inp["mask"]
    hx = inp["x"].cpu().pin_memory()
    hm = mask.cpu().pin_memory() if mask is not None else None
    hdy = inp["dy"].cpu().pin_memory()
    hy = torch.empty_like(hx).pin_memory()
    hdx = torch.empty_like(hx).pin_memory()
    d_x = torch.empty_like(inp["x"])
    d_m = torch.empty_like(mask) if hm is not None else None
    d_dy = torch.empty_like(inp["dy"])
    d_y = torch.empty_like(inp["x"])
    d_dx = torch.empty_like(inp["x"])
    hmf = hm.view(-1) if hm is not None else None
    dmf = d_m.view(-1) if d_m is not None else None
    dt = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}[hx.dtype]
    eb = hx.element_size()
    msb, msh = inp["mask_stride_b"], inp["mask_stride_h"]
    chunks = e2e_chunks(w, msb, msh, mask is not None)
    shared_mask = hm is not None and msb == 0  # one mask for every batch: copied in once per step
    s_in, s_k, s_out = (torch.cuda.Stream(device) for _ in range(3))
    ev_in = [torch.cuda.Event() for _ in chunks]
    ev_k = [torch.cuda.Event() for _ in chunks]
    ev_out = [torch.cuda.Event() for _ in chunks]
    ev_mask = torch.cuda.Event()

    def step():
        if shared_mask:
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_k[-1])  # the last block of the previous step has read it
                d_m.copy_(hm, non_blocking=True)
                ev_mask.record(s_in)
        for c, (r0, n, moff) in enumerate(chunks):
            r1 = r0 + n
            mlen = 0
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_k[c])  # the previous step's kernels are done with this block's inputs
                d_x[r0:r1].copy_(hx[r0:r1], non_blocking=True)
                d_dy[r0:r1].copy_(hdy[r0:r1], non_blocking=True)
                if hm is not None and not shared_mask:
                    nb = -(-n // (w.H * w.cols))
                    mlen = min(nb * msb, hmf.numel() - moff)
                    dmf[moff:moff + mlen].copy_(hmf[moff:moff + mlen], non_blocking=True)
                ev_in[c].record(s_in)
            s_k.wait_event(ev_in[c])
            s_k.wait_event(ev_out[c])  # the previous step's copy-out of this block has read y and dx
            if shared_mask:
                s_k.wait_event(ev_mask)
            st = s_k.cuda_stream
            mptr = None if d_m is None else d_m.data_ptr() + moff * d_m.element_size()
            mnum = 0 if d_m is None else (dmf.numel() - moff)
            rc = L.sms_forward(d_x.data_ptr() + r0 * w.cols * eb, mptr, mnum, msb, msh, inp["heads"],
                               d_y.data_ptr() + r0 * w.cols * eb, n, w.cols, w.scale, int(w.is_causal), dt, st)
            rc = rc or L.sms_backward(d_y.data_ptr() + r0 * w.cols * eb, d_dy.data_ptr() + r0 * w.cols * eb,
                                      d_dx.data_ptr() + r0 * w.cols * eb, n, w.cols, w.scale, int(w.is_causal),
                                      dt, st)
            if rc:
                raise RuntimeError(sms.sms_last_error())
            ev_k[c].record(s_k)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_k[c])
                hy[r0:r1].copy_(d_y[r0:r1], non_blocking=True)
                hdx[r0:r1].copy_(d_dx[r0:r1], non_blocking=True)
                ev_out[c].record(s_out)

    for _ in range(2):
        step()
    torch.cuda.synchronize(device)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for _ in range(steps):
        step()
    for s in (s_in, s_k):
        s_out.wait_stream(s)
    b.record(s_out)
    torch.cuda.synchronize(device)
    ms = a.elapsed_time(b) / steps
    # the same step with no overlap, for comparison: copies in, kernels, copies out
    a2, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    st0 = torch.cuda.current_stream(device)

    def serial_step():
        d_x.copy_(hx, non_blocking=True)
        if hm is not None:
            d_m.copy_(hm, non_blocking=True)
        d_dy.copy_(hdy, non_blocking=True)
        rc = L.sms_forward(d_x.data_ptr(), None if d_m is None else d_m.data_ptr(), 0 if d_m is None else d_m.numel(),
                           msb, msh, inp["heads"], d_y.data_ptr(), w.rows, w.cols, w.scale, int(w.is_causal), dt,
                           st0.cuda_stream)
        rc = rc or L.sms_backward(d_y.data_ptr(), d_dy.data_ptr(), d_dx.data_ptr(), w.rows, w.cols, w.scale,
                                  int(w.is_causal), dt, st0.cuda_stream)
        if rc:
            raise RuntimeError(sms.sms_last_error())
        hy.copy_(d_y, non_blocking=True)
        hdx.copy_(d_dx, non_blocking=True)

    serial_step()
    torch.cuda.synchronize(device)
    n2 = max(1, min(steps, 3))
    a2.record(st0)
    for _ in range(n2):
        serial_step()
    b2.record(st0)
    torch.cuda.synchronize(device)
    ms_serial = a2.elapsed_time(b2) / n2
    h2d = hx.numel() * eb + hdy.numel() * hdy.element_size() + (0 if hm is None else hm.numel() * hm.element_size())
    d2h = hy.numel() * hy.element_size() + hdx.numel() * hdx.element_size()
    alg = fwd_bytes(w, inp) + bwd_bytes(w)
    return {"value": round(alg / (ms * 1e6), 1), "unit": "GB/s", "ms_per_step": round(ms, 3),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "host_link_gbs": round((h2d + d2h) / (ms * 1e6), 1),
            "blocks": len(chunks), "serial_ms_per_step": round(ms_serial, 3),
            "path": "C ABI (sms_forward + sms_backward per row block) on pinned host buffers copied in and out "
                    "every step; copy-in, kernels and copy-out of successive blocks overlap on three streams"}


# ------------------------------------------------------ fused attention ---

ATTN_METRIC = "fused attention (QK^T, scaled masked softmax, PV) fwd/bwd achieved TFLOP/s and % of measured bf16 peak"


def attn_flops(B, H, S, D, causal):
    """Algorithmic FLOPs of one forward and one backward: 2 S S D per product
    per head (2 products forward, 5 backward); under causal only the
    S (S + 1) / 2 kept (query, key) pairs count."""
    pairs = S * (S + 1) / 2 if causal else S * S
    per = 2.0 * pairs * D * B * H
    return 2 * per, 5 * per


def _tc_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured (cuBLAS bf16 burst)"
    except Exception:
        return 1900.0, "fallback"


def run_attention(args, device):
    """The fused attention step on the tensor cores: forward (O, lse) and
    backward (dQ, dK, dV) through the C ABI on resident inputs."""
    import scaled_masked_softmax_gb300 as sms
    from scaled_masked_softmax_gb300 import workloads

    B, H, S, D = (int(v) for v in args.attn_shape.split(","))
    causal = not args.attn_no_causal
    dt = torch.bfloat16
    q, k, v, d_o = workloads.attention_inputs(B, H, S, D, "bf16", seed=41, device=device, with_do=True)
    mask, sb = None, 0
    if args.attn_mask:  # the [B,1,S,S] key padding of the bf16 S=4096 softmax workload, as bytes
        g = torch.Generator().manual_seed(42)
        L = torch.randint((S + 3) // 4, S + 1, (B,), generator=g)
        mask = (torch.arange(S)[None, :] >= L[:, None])[:, None, None, :].expand(B, 1, S, S).contiguous().to(device)
        sb = S * S
    L = sms.binding.lib()
    o = torch.empty_like(q)
    lse = torch.empty(B, H, S, dtype=torch.float32, device=device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    nws = sms.sms_attention_backward_workspace(B, H, S, D)
    ws = torch.empty(nws, dtype=torch.uint8, device=device)
    st = torch.cuda.current_stream(device).cuda_stream
    mptr = None if mask is None else mask.data_ptr()
    mnum = 0 if mask is None else mask.numel()
    scale = float(np.float32(1.0 / math.sqrt(D)))
    code = sms.SMS_BF16

    def fwd():
        rc = L.sms_attention_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), mptr, mnum, sb, 0, 1, o.data_ptr(),
                                     lse.data_ptr(), B, H, S, D, scale, int(causal), code, st)
        if rc:
            raise RuntimeError(sms.sms_last_error())

    def bwd():
        rc = L.sms_attention_backward(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), d_o.data_ptr(),
                                      lse.data_ptr(), mptr, mnum, sb, 0, 1, dq.data_ptr(), dk.data_ptr(),
                                      dv.data_ptr(), ws.data_ptr(), nws, B, H, S, D, scale, int(causal), code, st)
        if rc:
            raise RuntimeError(sms.sms_last_error())

    for _ in range(max(args.warmup, 3)):
        fwd()
        bwd()
    torch.cuda.synchronize(device)
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    clocks = ClockSampler(device)
    clocks.start()
    n0 = sms.sms_launch_count()
    for i in range(K):
        ev[i][0].record()
        fwd()
        ev[i][1].record()
        bwd()
        ev[i][2].record()
    torch.cuda.synchronize(device)
    n_launch = sms.sms_launch_count() - n0
    clk = clocks.stop()
    f_ms = statistics.mean(ev[i][0].elapsed_time(ev[i][1]) for i in range(K))
    b_ms = statistics.mean(ev[i][1].elapsed_time(ev[i][2]) for i in range(K))
    ff, bf = attn_flops(B, H, S, D, causal)
    peak, peak_kind = _tc_peak()
    tf = (ff + bf) / ((f_ms + b_ms) * 1e9)
    kern = {"forward": {"ms": round(f_ms, 4), "tflops": round(ff / (f_ms * 1e9), 1),
                        "frac_of_peak": round(ff / (f_ms * 1e9) / peak, 4)},
            "backward": {"ms": round(b_ms, 4), "tflops": round(bf / (b_ms * 1e9), 1),
                         "frac_of_peak": round(bf / (b_ms * 1e9) / peak, 4), "kernels": 3}}
    dom = "backward" if b_ms >= f_ms else "forward"
    res = {"metric": ATTN_METRIC, "value": round(tf, 1), "unit": "TFLOP/s", "n_gpus": 1, "steps": K,
           "warmup": args.warmup, "ms_per_step": round(f_ms + b_ms, 4), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded, workloads.attention_inputs)",
           "config": {"workload": f"attention_bf16_b{B}_h{H}_s{S}_d{D}" + ("_causal" if causal else "")
                      + ("_keypad" if mask is not None else ""),
                      "shape": [B, H, S, D], "is_causal": causal, "scale": scale,
                      "mask": "[B,1,S,S] key padding as bytes" if mask is not None else "none",
                      "step": "forward (O, lse) + backward (dQ, dK, dV)", "l2": "inputs larger than L2"
                      if 5 * q.numel() * 2 > L2_BYTES else "inputs fit in L2 (small shape)"},
           "kernels": kern,
           "roofline": {"kernel": dom, "bound": "tensor", "achieved": kern[dom]["tflops"], "peak": peak,
                        "unit": "TFLOP/s", "frac": kern[dom]["frac_of_peak"], "traffic": None,
                        "peak_source": peak_kind},
           "gpu_launches": int(n_launch), "clocks": clk}
    return res

# ------------------------------------------------------- oracle on the CPU ---

def _oracle_sample(w, inp_cpu, n_rows, start):
    import oracle

    rows = np.arange(start, start + n_rows, dtype=np.int64) % w.rows
    ti = torch.as_tensor(rows)
    xr = inp_cpu["x"][ti]
    y = oracle.forward(xr, w.cols, w.scale, w.is_causal, inp_cpu["mask"], inp_cpu["mask_stride_b"],
                       inp_cpu["mask_stride_h"], inp_cpu["heads"], row_index=rows)
    dyr = inp_cpu["dy"][ti]
    oracle.backward(y, dyr, w.cols, w.scale)
    return rows


_PER_ROW = {}


def _sample_bytes(w, rows_idx, inp_cpu):
    """Algorithmic bytes of forward + backward over the sampled rows: the GPU
    figure's per-row average (same accounting) times the rows processed."""
    if w.name not in _PER_ROW:
        _PER_ROW[w.name] = (fwd_bytes(w, inp_cpu) + bwd_bytes(w)) / w.rows
    return int(_PER_ROW[w.name] * len(rows_idx))


def cpu_inputs(w):
    from scaled_masked_softmax_gb300 import workloads

    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = workloads.make_inputs(w, device=dev, with_dy=True)
    return {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def run_cpu_baseline(w, inp_cpu, seconds):
    """Oracle throughput on the host cores over a time-bounded sample of rows."""
    import oracle

    oracle.build()
    cores = oracle.num_threads()
    chunk = max(64, min(4096, int(2_000_000 // w.cols)))
    t0 = time.perf_counter()
    done_bytes, n_rows, start = 0, 0, 0
    while True:
        idx = _oracle_sample(w, inp_cpu, chunk, start)
        done_bytes += _sample_bytes(w, idx, inp_cpu)
        n_rows += chunk
        start += chunk * 97  # spread the sample over the tensor
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    res = {"value": round(done_bytes / el / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
           "sample": f"{n_rows} rows of {w.name} (fwd+bwd, fp64, {chunk}-row chunks spread over the tensor), "
                     f"{el:.1f} s", "rows_per_s": round(n_rows / el, 1), "cpu": _cpu_model()}
    # the same oracle on one thread, over a shorter sample of the same rows
    prev = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        c1 = max(16, chunk // 8)
        t0 = time.perf_counter()
        b1, r1, start = 0, 0, 0
        while True:
            idx = _oracle_sample(w, inp_cpu, c1, start)
            b1 += _sample_bytes(w, idx, inp_cpu)
            r1 += c1
            start += c1 * 97
            el1 = time.perf_counter() - t0
            if el1 >= max(1.0, seconds / 4):
                break
    finally:
        oracle.set_num_threads(prev)
    res["single_thread"] = {"value": round(b1 / el1 / 1e9, 4), "unit": "GB/s", "rows_per_s": round(r1 / el1, 1),
                            "sample": f"{r1} rows, {el1:.1f} s"}
    return res


def _cpu_model() -> str:
    """The host CPU as /proc/cpuinfo names it (x86: model name; Arm: implementer and part codes)."""
    import platform

    name, impl, part = None, None, None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k, _, v = line.partition(":")
                k, v = k.strip(), v.strip()
                if k == "model name" and name is None:
                    name = v
                elif k == "CPU implementer" and impl is None:
                    impl = v
                elif k == "CPU part" and part is None:
                    part = v
    except OSError:
        pass
    if name:
        return name
    if impl or part:
        return f"{platform.machine()} implementer {impl} part {part}"
    return platform.machine()


def run_reference(args, rank, world):
    import oracle
    from scaled_masked_softmax_gb300 import workloads

    if rank != 0:
        return None
    w = _workload(args)
    inp_cpu = cpu_inputs(w)
    oracle.build()
    cores = oracle.num_threads()
    # size each step so the K timed steps take about a minute at most
    t = time.perf_counter()
    _oracle_sample(w, inp_cpu, 64, 0)
    per_row = (time.perf_counter() - t) / 64
    budget = max(5.0, min(60.0, 4.0 * args.steps))
    n = int(max(8, min(65536, budget / max(args.steps, 1) / max(per_row, 1e-7))))
    for i in range(max(args.warmup, 1)):
        _oracle_sample(w, inp_cpu, n, i * n)
    t0 = time.perf_counter()
    tot = 0
    for i in range(args.steps):
        idx = _oracle_sample(w, inp_cpu, n, (i + 7) * n * 13)
        tot += _sample_bytes(w, idx, inp_cpu)
    el = time.perf_counter() - t0
    value = tot / el / 1e9
    sample = f"{n} rows of {w.name} per step (fwd+bwd in fp64), {args.steps} steps"
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * el / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded, see workloads.py)",
        "config": {"workload": w.name, "rows": w.rows, "cols": w.cols, "mask": w.mask, "is_causal": w.is_causal,
                   "step": "forward + backward on a bounded row sample"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample, "cpu": _cpu_model()},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# -------------------------------------------------------------------- main ---

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--all", metavar="JSONL", default=None, help="also bench every workload into this file")
    ap.add_argument("--path", choices=["auto", "warp", "stream", "ring", "cta", "online"], default="auto",
                    help="force one kernel family (tuning); the default lets the dispatcher choose")
    ap.add_argument("--all-paths", action="store_true", help="with --all: every kernel family per workload")
    ap.add_argument("--only", default=None, help="with --all: comma-separated workload names")
    ap.add_argument("--graph", type=int, default=0, metavar="N",
                    help="also time the step replayed from a CUDA graph of N steps (launch-bound shapes)")
    ap.add_argument("--lengths", action="store_true",
                    help="key-padding workloads through the key-length entry points instead of the [B,1,S,S] mask")
    ap.add_argument("--bh", default=None, metavar="B,H",
                    help="the workload's distributions at batch B and H heads (small profiling captures)")
    ap.add_argument("--bool-mask", action="store_true",
                    help="masked workloads with the mask as one byte per element (sms_forward_bool)")
    ap.add_argument("--attention", action="store_true",
                    help="bench the fused attention step (tensor cores) instead of the softmax")
    ap.add_argument("--attn-shape", default="4,32,4096,128", metavar="B,H,S,D")
    ap.add_argument("--attn-no-causal", action="store_true")
    ap.add_argument("--attn-mask", action="store_true", help="with --attention: a [B,1,S,S] key-padding byte mask")
    args = ap.parse_args()

    world, rank, local = dist_env()
    init_dist(world, rank)

    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if rank == 0:
            print(json.dumps(res), flush=True)
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    if not torch.cuda.is_available():
        print(json.dumps({"metric": METRIC, "error": "no CUDA device"}))
        sys.exit(1)
    device = torch.device("cuda", local)
    import __graft_entry__

    __graft_entry__.build()
    import scaled_masked_softmax_gb300 as sms

    if args.attention:
        res = run_attention(args, device)
        print(json.dumps(res), flush=True)
        return
    path_code = {"auto": 0, "warp": 1, "cta": 2, "online": 3, "stream": 4, "ring": 5}
    sms.sms_set_forced_path(path_code[args.path])
    res, (w, inp, _y, _dx) = run_ours(args, rank, world, device)
    if rank == 0:
        # --e2e-steps 0 (profiling runs only) leaves the host-buffer leg out
        res["e2e"] = run_e2e(args, w, inp, device, args.e2e_steps) if args.e2e_steps > 0 else None
        if world == 1 and not args.no_cpu_baseline:
            res["cpu_baseline"] = run_cpu_baseline(w, {k: (v.cpu() if isinstance(v, torch.Tensor) else v)
                                                       for k, v in inp.items()}, args.cpu_seconds)
        else:
            res["cpu_baseline"] = None
    del inp, _y, _dx
    torch.cuda.empty_cache()
    if rank == 0:
        print(json.dumps(res), flush=True)
    if args.all and rank == 0 and world == 1:
        from scaled_masked_softmax_gb300 import workloads

        paths = ["auto", "warp", "stream", "ring", "cta", "online"] if args.all_paths else [args.path]
        with open(args.all, "w") as f:
            names = args.only.split(",") if args.only else list(workloads.WORKLOADS)
            for name in names:
                for pth in paths:
                    a2 = argparse.Namespace(**vars(args))
                    a2.workload = name
                    sms.sms_set_forced_path(path_code[pth])
                    try:
                        r, (w2, i2, y2, d2) = run_ours(a2, 0, 1, device)
                    except RuntimeError as e:  # the forced family cannot take this width
                        f.write(json.dumps({"workload": name, "path": pth, "skipped": str(e)}) + "\n")
                        torch.cuda.empty_cache()
                        continue
                    r.pop("clocks", None)
                    r["forced_path"] = pth
                    f.write(json.dumps(r) + "\n")
                    f.flush()
                    del i2, y2, d2
                    torch.cuda.empty_cache()
            sms.sms_set_forced_path(0)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
