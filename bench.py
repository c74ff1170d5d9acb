"""Benchmark of the exact-attention hot path on GB300.

One step = the whole path once over one batch of synthetic input: the
forward (fa_fwd) and the backward (fa_bwd: D preprocessing, the K/V-tile
main kernel, dQ conversion) at the headline shape B=4, H=16, N=8192, d=128,
bf16, causal.  The metric is attention TFLOPS, counting 4 B H N^2 d for the
forward (halved for causal) and 2.5x that for the backward.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Besides the contract keys the line carries, for the headline shape:
``l2_hot`` (the step again without the L2 flush), ``exp2_bound`` (the exp2
throughput probe and the exp-bound time of each direction),
``two_pass_bwd_leg``, ``window_leg``, ``varlen_leg`` and ``fp8_leg`` (the
deterministic backward, sliding window, packed batch and FP8 rows on their
own workloads), ``short_seq_leg`` (causal N = 512 and 1024, where both
directions run their persistent kernels), and ``configs_leg`` (forward and
backward of the tiny fp16, training, long-context and grouped-query
workloads; the fp64 oracle's host time on a bounded sample of each is in
``cpu_baseline.per_workload``); each can be switched off with its ``--no-*``
flag (``--no-configs`` covers the short-sequence leg too).

``--impl reference`` times the fp64 CPU oracle (test infrastructure, the
only other place this script runs it) on a bounded sample of the same
workload.  Under torchrun (N > 1) every rank processes its own batch shard
(weak scaling, no collective on the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd/bwd TFLOPS on 1 GB300 (bf16 d=128 N=8K causal); % of tensor peak"
L2_FLUSH_BYTES = 256 << 20


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None, help="workload name (default: the headline shape)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-two-pass", action="store_true", help="skip the deterministic two-pass backward leg")
    ap.add_argument("--no-window", action="store_true", help="skip the sliding-window leg")
    ap.add_argument("--no-varlen", action="store_true", help="skip the packed variable-length leg")
    ap.add_argument("--no-fp8", action="store_true", help="skip the FP8 leg (outlier workload)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload legs (tiny, training, long-context and grouped-query shapes)")
    return ap.parse_args()


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"bf16_tflops": p["bf16_tflops"], "bf16_tflops_sustained": p["bf16_tflops_sustained"],
                "hbm_gbs": p["hbm_gbs"], "source": "measured"}
    except Exception:
        return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0,
                "source": "fallback"}


def _src_sha(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "exact_attention_85_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _traffic(kernel: str, files):
    """DRAM bytes per launch from a committed ncu summary, if the kernel
    source is unchanged since that capture; else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic_bf16_b4_h16_n8k_causal.json")
    try:
        with open(path) as f:
            t = json.load(f)[kernel]
    except Exception:
        return None
    return t["bytes_per_launch"] if t.get("src_sha") == _src_sha(files) else None


class ClockSampler:
    """nvidia-smi samples taken while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), float(parts[2]), parts[3:7]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        loaded = [r for r in rows if r[2] > 300.0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(loaded)}


def run_ours(a):
    import torch

    from exact_attention_85_gb300 import _lib, attention_bwd, attention_fwd
    from exact_attention_85_gb300.inputs import HEADLINE, WORKLOADS, make_inputs

    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = WORKLOADS[a.workload or HEADLINE]
    lib = _lib.load()
    stream = torch.cuda.current_stream()

    # weak scaling: the global problem has B * ws batches; this rank owns the
    # contiguous (batch, kv-head) units of its own B batches (no exchange)
    from exact_attention_85_gb300.sharding import unit_range
    u_lo, u_hi = unit_range(w.B * ws, w.Hkv, ws, rank)
    assert u_hi - u_lo == w.B * w.Hkv
    host = make_inputs(w, seed=w.seed + 1000 * rank, with_grad=True)
    q, k, v, dO = (host[n].to(dev).contiguous() for n in ("q", "k", "v", "dO"))
    B, Hq, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_bytes = _lib.fa_bwd_workspace_bytes(B, Hq, N, d)
    workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def fwd():
        _lib.fa_fwd(q, k, v, o, lse, w.causal, w.scale, stream)

    def bwd():
        _lib.fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, w.causal, w.scale, workspace, stream)

    has_bwd = w.backward
    if has_bwd:
        fwd()
        bwd()  # any failure raises: a step without its backward is not a step
    for _ in range(a.warmup):
        fwd()
        if has_bwd:
            bwd()
        flush.zero_()
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(a.steps)]
    launches = 0
    with ClockSampler(torch.cuda.current_device()) as clk:
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(a.steps):
            ev[i][0].record(stream)
            fwd()
            launches += 1
            ev[i][1].record(stream)
            if has_bwd:
                bwd()
                launches += 3
            ev[i][2].record(stream)
            flush.zero_()  # L2 flush between steps, outside the events
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    if ws > 1:
        torch.distributed.barrier()
    status = _lib.fa_get_device_status(stream)
    if status != _lib.FA_OK:
        raise RuntimeError("a bounded device wait ran out during the timed region")

    fwd_ms = [e[0].elapsed_time(e[1]) for e in ev]
    bwd_ms = [e[1].elapsed_time(e[2]) for e in ev] if has_bwd else [0.0] * a.steps
    step_ms = statistics.mean(f + b for f, b in zip(fwd_ms, bwd_ms))
    if ws > 1:
        t = torch.tensor([step_ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        step_ms = float(t.item())

    f_fwd = w.fwd_flops()
    f_bwd = w.bwd_flops() if has_bwd else 0.0
    value = ws * (f_fwd + f_bwd) / (step_ms * 1e-3) / 1e12
    peaks = _peaks()
    fwd_avg = statistics.mean(fwd_ms)
    bwd_avg = statistics.mean(bwd_ms) if has_bwd else 0.0
    fwd_tf = f_fwd / (fwd_avg * 1e-3) / 1e12
    bwd_tf = f_bwd / (bwd_avg * 1e-3) / 1e12 if has_bwd else None

    # roofline of the dominant kernel (the longer of the two timed calls)
    if has_bwd and bwd_avg > fwd_avg:
        dom, dom_ms, dom_flops = "fa_bwd (main kernel; duration includes the small D and dQ-convert kernels)", bwd_avg, f_bwd
        traffic = _traffic("bwd_kernel", ["fa_bwd.cu", "grid_order.cuh"])
    else:
        dom, dom_ms, dom_flops = "fwd_kernel", fwd_avg, f_fwd
        traffic = _traffic("fwd_kernel", ["fa_fwd.cu", "grid_order.cuh"])
    achieved = dom_flops / (dom_ms * 1e-3) / 1e12
    roof = {"kernel": dom, "bound": "tensor", "achieved": round(achieved, 1), "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4), "traffic": traffic,
            "peak_source": f"{peaks['source']} bf16 burst (kernel timed alone with CUDA events)"}

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "TFLOPS", "n_gpus": ws, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": round(step_ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "N": w.N, "d": w.d,
                   "causal": w.causal, "per_gpu_batch": w.B, "global_batch": w.B * ws,
                   "parallelism": f"dp{ws} (batch shards, no collective)",
                   "units_rank0": [u_lo, u_hi] if rank == 0 else None,
                   "l2": "flushed between steps (256 MB write); inputs 537 MB also exceed L2; "
                         "l2_hot repeats the timing without the flush",
                   "backward_included": has_bwd},
        "fwd_ms": round(fwd_avg, 4), "bwd_ms": round(bwd_avg, 4),
        "fwd_tflops": round(fwd_tf, 1), "bwd_tflops": None if bwd_tf is None else round(bwd_tf, 1),
        "fwd_frac_of_peak": round(fwd_tf / peaks["bf16_tflops"], 4),
        "bwd_frac_of_peak": None if bwd_tf is None else round(bwd_tf / peaks["bf16_tflops"], 4),
        "roofline": roof, "gpu_launches": launches, "wall_s_timed": round(wall, 3),
        "clocks": clk.summary(),
    }

    result["l2_hot"] = _hot_leg(a, fwd, bwd if has_bwd else None, stream, f_fwd, f_bwd)
    result["exp2_bound"] = _exp2_leg(w, dev, stream, fwd_avg, bwd_avg if has_bwd else None)

    if has_bwd and not a.no_two_pass:
        result["two_pass_bwd_leg"] = _two_pass_leg(a, w, (q, k, v, o, lse, dO, dq, dk, dv), dev, stream, peaks,
                                                   flush)
    if has_bwd and not a.no_window and w.causal:
        result["window_leg"] = _window_leg(a, w, (q, k, v, o, lse, dO, dq, dk, dv), dev, stream, peaks, flush)
    if has_bwd and not a.no_varlen and a.workload is None:
        result["varlen_leg"] = _varlen_leg(a, dev, stream, peaks, flush)
    if not a.no_fp8 and a.workload is None:
        result["fp8_leg"] = _fp8_leg(a, dev, stream, peaks)
    if not a.no_configs and a.workload is None:
        result["configs_leg"] = _configs_leg(a, dev, stream, peaks, flush)
        result["short_seq_leg"] = _short_leg(a, dev, stream, peaks, flush)
    if not a.no_e2e:
        result["e2e"] = _e2e(a, w, host, dev, stream, has_bwd, ws)
    if rank == 0 and ws == 1 and not a.no_cpu:
        result["cpu_baseline"] = _cpu_baseline(w, host, budget_s=12.0)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def _hot_leg(a, fwd, bwd, stream, f_fwd, f_bwd):
    """The same calls back to back with no L2 flush between them (inputs
    partly L2-resident from the previous call)."""
    import torch

    for _ in range(2):
        fwd()
        if bwd:
            bwd()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(a.steps)]
    torch.cuda.synchronize()
    for i in range(a.steps):
        ev[i][0].record(stream)
        fwd()
        ev[i][1].record(stream)
        if bwd:
            bwd()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    fm = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    out = {"l2": "not flushed between steps", "fwd_ms": round(fm, 4),
           "fwd_tflops": round(f_fwd / (fm * 1e-3) / 1e12, 1), "launches_per_step": 4 if bwd else 1}
    if bwd:
        bm = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
        out.update(bwd_ms=round(bm, 4), bwd_tflops=round(f_bwd / (bm * 1e-3) / 1e12, 1))
    return out


def _visible_pairs(w) -> float:
    """(query, key) pairs the mask lets through, over all heads and batches."""
    per = w.N * (w.N + 1) / 2 if w.causal else w.N * w.N
    return float(w.B * w.Hq * per)


def _exp2_leg(w, dev, stream, fwd_ms, bwd_ms):
    """exp2 throughput of the special-function unit (fa_probe_exp2) and the
    time the forward / backward would take if bound by their exps alone:
    one exp per visible score in the forward, one more per score in the
    backward's recomputation of P."""
    import torch
    from exact_attention_85_gb300 import _lib

    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    blocks, iters = sms * 8, 2048
    sink = torch.empty(blocks * 256, dtype=torch.float32, device=dev)
    for _ in range(3):
        n = _lib.fa_probe_exp2(sink, blocks, iters, stream)
    times = []
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        n = _lib.fa_probe_exp2(sink, blocks, iters, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    ms = statistics.median(times)
    rate = n / (ms * 1e-3)
    exps = _visible_pairs(w)
    out = {"probe": f"{blocks} blocks x 256 threads x 8 chains x {iters} ex2.approx.ftz.f32", "probe_ms": round(ms, 4),
           "exp2_per_s": float(f"{rate:.4g}"), "exps_fwd": exps, "fwd_exp_bound_ms": round(exps / rate * 1e3, 4),
           "fwd_exp_share": round(exps / rate * 1e3 / fwd_ms, 3), "launches": 8}
    if bwd_ms:
        out.update(exps_bwd=exps, bwd_exp_bound_ms=round(exps / rate * 1e3, 4),
                   bwd_exp_share=round(exps / rate * 1e3 / bwd_ms, 3))
    return out


def _two_pass_leg(a, w, t, dev, stream, peaks, flush):
    """The deterministic two-pass backward (fa_bwd_two_pass) on the step's
    workload, timed like the step's backward.  TFLOPS count the same five
    matrix products as fa_bwd; the two-pass form executes seven (S and dP are
    formed once in each pass)."""
    import torch

    from exact_attention_85_gb300 import _lib

    q, k, v, o, lse, dO, dq, dk, dv = t
    B, Hq, N, d = q.shape
    ws = torch.empty(_lib.fa_bwd_two_pass_workspace_bytes(B, Hq, N, d), dtype=torch.uint8, device=dev)

    def bwd():
        _lib.fa_bwd_two_pass(q, k, v, o, lse, dO, dq, dk, dv, w.causal, w.scale, ws, stream)

    for _ in range(max(3, a.warmup)):
        bwd()
        flush.zero_()
    torch.cuda.synchronize()
    steps = max(3, min(a.steps, 10))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for i in range(steps):
        ev[i][0].record(stream)
        bwd()
        ev[i][1].record(stream)
        flush.zero_()
    torch.cuda.synchronize()
    if _lib.fa_get_device_status(stream) != _lib.FA_OK:
        raise RuntimeError("a bounded device wait ran out during the two-pass backward leg")
    ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    tf = w.bwd_flops() / (ms * 1e-3) / 1e12
    return {"workload": w.name, "bwd_ms": round(ms, 4), "bwd_tflops": round(tf, 1),
            "bwd_frac_of_peak": round(tf / peaks["bf16_tflops"], 4),
            "executed_tflops": round(tf * 7.0 / 5.0, 1), "launches_per_step": 3, "deterministic": True}


def _window_leg(a, w, t, dev, stream, peaks, flush, window=1024):
    """Causal sliding-window attention (fa_fwd_local / fa_bwd_local, atomic
    dQ) on the step's workload with a window of `window` keys.  FLOPs count
    the visible (query, key) pairs only: sum over rows of min(r + 1, W)."""
    import torch

    from exact_attention_85_gb300 import _lib

    q, k, v, o, lse, dO, dq, dk, dv = t
    B, Hq, N, d = q.shape
    ws = torch.empty(_lib.fa_bwd_workspace_bytes(B, Hq, N, d), dtype=torch.uint8, device=dev)
    W = min(window, N)
    pairs = W * (W + 1) / 2 + (N - W) * W
    f_fwd = 4.0 * B * Hq * d * pairs
    f_bwd = 2.5 * f_fwd

    def fwd():
        _lib.fa_fwd_local(q, k, v, o, lse, W, w.scale, stream)

    def bwd():
        _lib.fa_bwd_local(q, k, v, o, lse, dO, dq, dk, dv, W, w.scale, False, ws, stream)

    for _ in range(max(3, a.warmup)):
        fwd()
        bwd()
        flush.zero_()
    torch.cuda.synchronize()
    steps = max(3, min(a.steps, 10))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for i in range(steps):
        ev[i][0].record(stream)
        fwd()
        ev[i][1].record(stream)
        bwd()
        ev[i][2].record(stream)
        flush.zero_()
    torch.cuda.synchronize()
    if _lib.fa_get_device_status(stream) != _lib.FA_OK:
        raise RuntimeError("a bounded device wait ran out during the sliding-window leg")
    f_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    b_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    ftf = f_fwd / (f_ms * 1e-3) / 1e12
    btf = f_bwd / (b_ms * 1e-3) / 1e12
    return {"workload": f"{w.name} window={W}", "fwd_ms": round(f_ms, 4), "bwd_ms": round(b_ms, 4),
            "fwd_tflops": round(ftf, 1), "bwd_tflops": round(btf, 1),
            "fwd_frac_of_peak": round(ftf / peaks["bf16_tflops"], 4),
            "bwd_frac_of_peak": round(btf / peaks["bf16_tflops"], 4), "launches_per_step": 4,
            "flops": "visible (query, key) pairs only"}


def _varlen_leg(a, dev, stream, peaks, flush, n_seq=8, max_len=8192, Hq=16, d=128):
    """Packed variable-length batch (fa_fwd_varlen / fa_bwd_varlen, atomic dQ):
    a seeded mix of 8 causal bf16 sequences of 1 .. 8192 rows, H16 d128,
    token-major.  FLOPs count each sequence's own causal pairs n (n + 1) / 2."""
    import torch

    from exact_attention_85_gb300 import _lib
    from exact_attention_85_gb300.inputs import make_varlen, varlen_lengths

    lengths = varlen_lengths(n_seq, max_len, seed=11)
    x = make_varlen(lengths, Hq, Hq, d, torch.bfloat16, seed=12)
    q, k, v, dO = (x[n].to(dev).contiguous() for n in ("q", "k", "v", "dO"))
    cu = x["cu_seqlens"].to(dev)
    total = q.shape[0]
    o = torch.empty_like(q)
    lse = torch.empty((Hq, total), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(_lib.fa_bwd_varlen_workspace_bytes(total, Hq, d, False), dtype=torch.uint8, device=dev)
    mx = max(lengths)
    scale = d ** -0.5
    pairs = sum(n * (n + 1) / 2 for n in lengths)
    f_fwd = 4.0 * Hq * d * pairs
    f_bwd = 2.5 * f_fwd

    def fwd():
        _lib.fa_fwd_varlen(q, k, v, o, lse, cu, mx, True, scale, 0, stream)

    def bwd():
        _lib.fa_bwd_varlen(q, k, v, o, lse, dO, dq, dk, dv, cu, mx, True, scale, False, ws, 0, stream)

    for _ in range(max(3, a.warmup)):
        fwd()
        bwd()
        flush.zero_()
    torch.cuda.synchronize()
    steps = max(3, min(a.steps, 10))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for i in range(steps):
        ev[i][0].record(stream)
        fwd()
        ev[i][1].record(stream)
        bwd()
        ev[i][2].record(stream)
        flush.zero_()
    torch.cuda.synchronize()
    if _lib.fa_get_device_status(stream) != _lib.FA_OK:
        raise RuntimeError("a bounded device wait ran out during the packed-batch leg")
    f_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    b_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    ftf = f_fwd / (f_ms * 1e-3) / 1e12
    btf = f_bwd / (b_ms * 1e-3) / 1e12
    return {"workload": f"packed bf16 H{Hq} d{d} causal, lengths {lengths} (total {total})",
            "fwd_ms": round(f_ms, 4), "bwd_ms": round(b_ms, 4), "fwd_tflops": round(ftf, 1),
            "bwd_tflops": round(btf, 1), "fwd_frac_of_peak": round(ftf / peaks["bf16_tflops"], 4),
            "bwd_frac_of_peak": round(btf / peaks["bf16_tflops"], 4), "launches_per_step": 4,
            "flops": "each sequence's causal pairs only"}


def _fp8_leg(a, dev, stream, peaks):
    """The FP8 rows of the path on their own workload (B4 H16 N8192 d128,
    non-causal, 0.1% outliers): random-sign Hadamard + e4m3 quantisation of
    Q and K, plain quantisation of V, then the FP8 forward.  Reported beside
    the bf16 step, not part of it."""
    import torch

    from exact_attention_85_gb300 import _lib
    from exact_attention_85_gb300.inputs import WORKLOADS, make_inputs

    w = WORKLOADS["fp8_b4_h16_n8k_outliers"]
    host = make_inputs(w, with_grad=False)
    q, k, v = (host[n].to(dev).contiguous() for n in ("q", "k", "v"))
    signs = host["signs"].to(dev)
    B, Hq, N, d = q.shape
    q8, k8, v8 = (torch.empty(t.shape, dtype=torch.uint8, device=dev) for t in (q, k, v))
    ds = torch.empty(3, dtype=torch.float32, device=dev)
    ws = torch.empty(3 * 256, dtype=torch.uint8, device=dev)
    o = torch.empty((B, Hq, N, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def quant():
        _lib.fa_hadamard_quant_fp8(q, signs, q8, ds[0:1], ws[0:256], stream)
        _lib.fa_hadamard_quant_fp8(k, signs, k8, ds[1:2], ws[256:512], stream)
        _lib.fa_hadamard_quant_fp8(v, None, v8, ds[2:3], ws[512:768], stream)

    def fwd():
        _lib.fa_fwd_fp8(q8, k8, v8, ds[0:1], ds[1:2], ds[2:3], o, lse, w.causal, w.scale, stream)

    for _ in range(max(3, a.warmup)):
        quant()
        fwd()
        flush.zero_()
    torch.cuda.synchronize()
    steps = max(3, min(a.steps, 10))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for i in range(steps):
        ev[i][0].record(stream)
        quant()
        ev[i][1].record(stream)
        fwd()
        ev[i][2].record(stream)
        flush.zero_()
    torch.cuda.synchronize()
    if _lib.fa_get_device_status(stream) != _lib.FA_OK:
        raise RuntimeError("a bounded device wait ran out during the FP8 leg")
    q_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    f_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    tflops = w.fwd_flops() / (f_ms * 1e-3) / 1e12

    # the same FP8 operands with the causal mask (half the FLOPs)
    def fwd_causal():
        _lib.fa_fwd_fp8(q8, k8, v8, ds[0:1], ds[1:2], ds[2:3], o, lse, True, w.scale, stream)

    for _ in range(3):
        fwd_causal()
    torch.cuda.synchronize()
    evc = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for i in range(steps):
        evc[i][0].record(stream)
        fwd_causal()
        evc[i][1].record(stream)
        flush.zero_()
    torch.cuda.synchronize()
    c_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evc)
    c_tflops = w.fwd_flops() / 2 / (c_ms * 1e-3) / 1e12
    fp8_peak = 2.0 * peaks["bf16_tflops"]
    q_bytes = 3 * q.numel() * (2 + 1)  # algorithmic: read bf16 once, write e4m3 once
    return {"workload": w.name, "fwd_ms": round(f_ms, 4), "fwd_tflops": round(tflops, 1),
            "fwd_frac_of_fp8_peak": round(tflops / fp8_peak, 4),
            "fp8_peak": fp8_peak, "fp8_peak_source": f"2 x {peaks['source']} bf16 burst (nominal FP8/BF16 ratio)",
            "fwd_causal_ms": round(c_ms, 4), "fwd_causal_tflops": round(c_tflops, 1),
            "quant_ms_3_tensors": round(q_ms, 4),
            "quant_gbs_algorithmic": round(q_bytes / (q_ms * 1e-3) / 1e9, 1),
            "quant_frac_of_hbm": round(q_bytes / (q_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
            "launches_per_step": 3 * 3 + 1}


CONFIG_LEGS = ("tiny_fp16_d64_n256", "train_bf16_b8_h16_n2k_causal", "long_bf16_b1_h16_n16k_causal",
               "gqa_bf16_b4_hq32_hkv8_n4k_causal")
# short sequences (bf16, d = 128, 16 heads, causal), where fa_fwd and fa_bwd
# run their persistent kernels: (B, N)
SHORT_LEGS = ((32, 512), (16, 1024))


def _configs_leg(a, dev, stream, peaks, flush):
    """Forward and backward (fa_fwd, fa_bwd) of each workload in CONFIG_LEGS,
    timed like the step (CUDA events per call, L2 flushed between steps).
    The fp64 oracle's host time for each of them is in
    cpu_baseline.per_workload."""
    import torch

    from exact_attention_85_gb300 import _lib
    from exact_attention_85_gb300.inputs import WORKLOADS, make_inputs

    out = {}
    for name in CONFIG_LEGS:
        w = WORKLOADS[name]
        host = make_inputs(w, with_grad=True)
        q, k, v, dO = (host[n].to(dev).contiguous() for n in ("q", "k", "v", "dO"))
        B, Hq, N, d = q.shape
        o = torch.empty_like(q)
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        wsb = torch.empty(_lib.fa_bwd_workspace_bytes(B, Hq, N, d), dtype=torch.uint8, device=dev)

        def fwd():
            _lib.fa_fwd(q, k, v, o, lse, w.causal, w.scale, stream)

        def bwd():
            _lib.fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, w.causal, w.scale, wsb, stream)

        for _ in range(max(3, a.warmup)):
            fwd()
            bwd()
            flush.zero_()
        torch.cuda.synchronize()
        steps = max(3, min(a.steps, 20))
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
        for i in range(steps):
            ev[i][0].record(stream)
            fwd()
            ev[i][1].record(stream)
            bwd()
            ev[i][2].record(stream)
            flush.zero_()
        torch.cuda.synchronize()
        if _lib.fa_get_device_status(stream) != _lib.FA_OK:
            raise RuntimeError(f"a bounded device wait ran out during the {name} leg")
        f_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
        b_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
        ftf = w.fwd_flops() / (f_ms * 1e-3) / 1e12
        btf = w.bwd_flops() / (b_ms * 1e-3) / 1e12
        # the persistent forward (fa_fwd_persistent) on the same inputs
        for _ in range(3):
            _lib.fa_fwd_persistent(q, k, v, o, lse, w.causal, w.scale, stream)
        torch.cuda.synchronize()
        evp = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        for i in range(steps):
            evp[i][0].record(stream)
            _lib.fa_fwd_persistent(q, k, v, o, lse, w.causal, w.scale, stream)
            evp[i][1].record(stream)
            flush.zero_()
        torch.cuda.synchronize()
        if _lib.fa_get_device_status(stream) != _lib.FA_OK:
            raise RuntimeError(f"a bounded device wait ran out during the {name} leg (persistent forward)")
        p_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evp)
        ptf = w.fwd_flops() / (p_ms * 1e-3) / 1e12
        leg = {"B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "N": w.N, "d": w.d, "dtype": w.dtype, "causal": w.causal,
               "fwd_persistent_ms": round(p_ms, 4), "fwd_persistent_tflops": round(ptf, 1),
               "fwd_ms": round(f_ms, 4), "bwd_ms": round(b_ms, 4), "fwd_tflops": round(ftf, 1),
               "bwd_tflops": round(btf, 1), "fwd_frac_of_peak": round(ftf / peaks["bf16_tflops"], 4),
               "bwd_frac_of_peak": round(btf / peaks["bf16_tflops"], 4), "launches_per_step": 4}
        out[name] = leg
        del q, k, v, dO, o, lse, dq, dk, dv, wsb
    return out


def _short_leg(a, dev, stream, peaks, flush):
    """fa_fwd / fa_bwd at short causal lengths (SHORT_LEGS), where both run
    their persistent kernels, timed like the step (L2 flushed between
    steps)."""
    import torch

    from exact_attention_85_gb300 import _lib
    from exact_attention_85_gb300.inputs import make_custom

    out = {}
    for B, N in SHORT_LEGS:
        H, d = 16, 128
        x = make_custom(B, H, H, N, d, torch.bfloat16, seed=N)
        q, k, v, dO = (x[n].to(dev).contiguous() for n in ("q", "k", "v", "dO"))
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        wsb = torch.empty(_lib.fa_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=dev)
        scale = d ** -0.5
        for _ in range(max(3, a.warmup)):
            _lib.fa_fwd(q, k, v, o, lse, True, scale, stream)
            _lib.fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, True, scale, wsb, stream)
        torch.cuda.synchronize()
        steps = max(3, min(a.steps, 20))
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
        for i in range(steps):
            ev[i][0].record(stream)
            _lib.fa_fwd(q, k, v, o, lse, True, scale, stream)
            ev[i][1].record(stream)
            _lib.fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, True, scale, wsb, stream)
            ev[i][2].record(stream)
            flush.zero_()
        torch.cuda.synchronize()
        if _lib.fa_get_device_status(stream) != _lib.FA_OK:
            raise RuntimeError(f"a bounded device wait ran out during the short-sequence leg (N={N})")
        f_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
        b_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
        f_fl = 2.0 * B * H * N * N * d
        out[f"bf16_b{B}_h{H}_n{N}_causal"] = {
            "fwd_ms": round(f_ms, 4), "bwd_ms": round(b_ms, 4),
            "fwd_tflops": round(f_fl / (f_ms * 1e-3) / 1e12, 1), "bwd_tflops": round(2.5 * f_fl / (b_ms * 1e-3) / 1e12, 1),
            "fwd_frac_of_peak": round(f_fl / (f_ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
            "bwd_frac_of_peak": round(2.5 * f_fl / (b_ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
            "kernels": "persistent forward and persistent backward main kernel", "launches_per_step": 4}
        del q, k, v, dO, o, lse, dq, dk, dv, wsb
    return out


def _e2e(a, w, host, dev, stream, has_bwd, ws):
    """Same metric through the public API with pinned host buffers: every step
    copies Q, K, V, dO in and O, dQ, dK, dV out inside the timed region.  The
    copies run on their own streams, double-buffered, so step i's kernels
    overlap the copy-in of step i + 1 and the copy-out of step i - 1 (the usual
    way to feed a GPU from host memory); the forward starts once Q, K, V are
    in (dO follows) and O goes out as soon as the forward is done.  The timed
    region spans from before the first copy-in to after the last copy-out,
    over the same K steps as the device-side timing."""
    import torch

    from exact_attention_85_gb300 import attention_bwd, attention_fwd

    names_in = ("q", "k", "v", "dO")
    names_out = ("o", "dq", "dk", "dv") if has_bwd else ("o",)
    h_in = {n: host[n].pin_memory() for n in names_in}
    like = {"o": "q", "dq": "q", "dk": "k", "dv": "v"}
    h_out = [{n: torch.empty_like(host[like[n]]).pin_memory() for n in names_out} for _ in range(2)]
    d_in = [{n: torch.empty(h_in[n].shape, dtype=h_in[n].dtype, device=dev) for n in names_in} for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_qkv = [torch.cuda.Event() for _ in range(2)]  # Q, K, V of buffer set s are in
    ev_in = [torch.cuda.Event() for _ in range(2)]  # and dO
    ev_fwd = [torch.cuda.Event() for _ in range(2)]  # the forward of the step that used set s is done
    ev_done = [torch.cuda.Event() for _ in range(2)]  # kernels of the step that used buffer set s
    ev_out = [torch.cuda.Event() for _ in range(2)]
    steps = max(3, a.steps)

    def run(n_steps):
        for i in range(n_steps):
            s = i & 1
            # copy-in to buffer set s once the kernels of step i - 2 are done with it
            if i >= 2:
                s_in.wait_event(ev_done[s])
            with torch.cuda.stream(s_in):
                for n in names_in:
                    d_in[s][n].copy_(h_in[n], non_blocking=True)
                    if n == "v":
                        ev_qkv[s].record(s_in)
                ev_in[s].record(s_in)
            stream.wait_event(ev_qkv[s])
            x = d_in[s]
            o, lse = attention_fwd(x["q"], x["k"], x["v"], w.causal, w.scale, stream)
            ev_fwd[s].record(stream)
            outs = {}
            if has_bwd:
                stream.wait_event(ev_in[s])
                dq, dk, dv = attention_bwd(x["q"], x["k"], x["v"], o, lse, x["dO"], w.causal, w.scale,
                                           stream=stream)
                outs.update(dq=dq, dk=dk, dv=dv)
            ev_done[s].record(stream)
            # copy-out of this step's results, O as soon as the forward is
            # done (host set s is free once the copy-out of step i - 2 has
            # finished: same stream, in order)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_fwd[s])
                o.record_stream(s_out)
                h_out[s]["o"].copy_(o, non_blocking=True)
                s_out.wait_event(ev_done[s])
                for n, t in outs.items():
                    t.record_stream(s_out)
                    h_out[s][n].copy_(t, non_blocking=True)
                ev_out[s].record(s_out)
        stream.wait_stream(s_out)
        stream.wait_stream(s_in)

    run(2)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run(steps)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    if ws > 1:
        t = torch.tensor([ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
    flops = w.fwd_flops() + (w.bwd_flops() if has_bwd else 0.0)
    h2d = sum(h_in[n].numel() * h_in[n].element_size() for n in names_in)
    d2h = sum(t.numel() * t.element_size() for t in h_out[0].values())
    return {"value": round(ws * flops / (ms * 1e-3) / 1e12, 1), "unit": "TFLOPS", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "overlap": "copy-in of step i+1 and copy-out of step i-1 on their own streams during step i; "
                       "the forward starts once Q, K, V are in, O goes out after the forward"}


def _cpu_sample(w, host, n_groups: int):
    """fp64 oracle forward + backward of the first `n_groups` (batch, kv-head)
    groups at full sequence length; returns (seconds, algorithmic flops)."""
    import oracle

    G = w.Hq // w.Hkv
    t0 = time.perf_counter()
    done = 0
    for idx in range(n_groups):
        b, g = divmod(idx, w.Hkv)
        sl_q = slice(g * G, g * G + G)
        oracle.attention_bwd_group(host["q"][b:b + 1, sl_q], host["k"][b:b + 1, g:g + 1],
                                   host["v"][b:b + 1, g:g + 1], host["dO"][b:b + 1, sl_q],
                                   0, 0, w.causal, w.scale)
        done += G
    secs = time.perf_counter() - t0
    per_head = (w.fwd_flops() + w.bwd_flops()) / (w.B * w.Hq)
    return secs, per_head * done


def _cpu_single_thread_small():
    """The oracle on one host thread, forward + backward of the whole small
    fp16 workload (B1 H2 N256 d64, non-causal)."""
    import oracle
    from exact_attention_85_gb300.inputs import WORKLOADS, make_inputs

    w1 = WORKLOADS["tiny_fp16_d64_n256"]
    host1 = make_inputs(w1, with_grad=True)
    oracle.set_threads(1)
    try:
        _cpu_sample(w1, host1, w1.B * w1.Hkv)  # warm-up (library load)
        reps, secs, flops = 0, 0.0, 0.0
        while secs < 1.0:
            s1, f1 = _cpu_sample(w1, host1, w1.B * w1.Hkv)
            secs, flops, reps = secs + s1, flops + f1, reps + 1
    finally:
        oracle.set_threads(0)
    return {"workload": w1.name, "value": round(flops / secs / 1e12, 6), "unit": "TFLOPS", "cores": 1,
            "ms_per_step": round(1e3 * secs / reps, 3), "sample": f"{reps} fwd+bwd passes of the whole workload"}


def _cpu_baseline(w, host, budget_s: float):
    threads = os.cpu_count() or 1
    secs, flops = _cpu_sample(w, host, 1)
    n = 1
    if secs < budget_s / 2:
        extra = max(0, int(budget_s / max(secs, 1e-3)) - 1)
        if extra:
            s2, f2 = _cpu_sample(w, host, min(extra, w.B * w.Hkv))
            secs, flops, n = secs + s2, flops + f2, 1 + min(extra, w.B * w.Hkv)
    return {"value": round(flops / secs / 1e12, 6), "unit": "TFLOPS", "cores": threads, "kind": "oracle",
            "sample": f"fp64 oracle forward+backward of {n} (batch, kv-head) group(s) of {w.name} at full "
                      f"N={w.N}, {secs:.1f} s, OpenMP over {threads} host threads",
            "single_thread": _cpu_single_thread_small(),
            "per_workload": _cpu_per_workload()}


def _cpu_per_workload():
    """The oracle (all host threads) on a bounded sample of each workload of
    the per-workload legs: one (batch, kv-head) group at full N, or the whole
    workload when it is that small."""
    from exact_attention_85_gb300.inputs import WORKLOADS, make_inputs

    out = {}
    for name in CONFIG_LEGS:
        w = WORKLOADS[name]
        host = make_inputs(w, with_grad=True)
        groups = w.B * w.Hkv if w.N <= 256 else 1
        secs, flops = _cpu_sample(w, host, groups)
        out[name] = {"tflops": round(flops / secs / 1e12, 6), "seconds": round(secs, 3),
                     "cores": os.cpu_count() or 1,
                     "sample": f"fp64 forward+backward of {groups} (batch, kv-head) group(s) at full N={w.N}"}
    return out


def run_reference(a):
    """The fp64 CPU oracle as the reference arm (rank 0 only)."""
    ws, rank, _ = _dist()
    if rank != 0:
        return
    from exact_attention_85_gb300.inputs import HEADLINE, WORKLOADS, make_inputs
    w = WORKLOADS[a.workload or HEADLINE]
    host = make_inputs(w, with_grad=True)
    threads = os.cpu_count() or 1
    for _ in range(a.warmup):
        _cpu_sample(w, host, 1)
    times, flops = [], 0.0
    for i in range(a.steps):
        s, f = _cpu_sample(w, host, 1)
        times.append(s)
        flops = f
    ms = statistics.mean(times) * 1e3
    value = flops / (ms * 1e-3) / 1e12
    out = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOPS", "n_gpus": ws,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(ms, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "N": w.N, "d": w.d,
                   "causal": w.causal, "sample_per_step": "one (batch, kv-head) group at full N"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOPS", "cores": threads, "kind": "oracle",
                         "sample": "each step: fp64 oracle forward+backward of one (batch, kv-head) group at "
                                   f"full N={w.N}"},
        "e2e": {"value": round(value, 6), "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


if __name__ == "__main__":
    args = _args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)
