"""Host-side checks of the benchmark script: the reference arm's JSON line
(it times the fp64 oracle, so it runs without a GPU) and the FLOP / exp
counting helpers the GPU legs use."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOPS" and d["higher_is_better"] is True
    assert d["steps"] == 1 and d["warmup"] == 0 and d["n_gpus"] == 1 and d["dtype"] == "f64"
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["workload"] == "bf16_b4_h16_n8k_d128_causal"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_visible_pairs_and_flop_counts():
    import bench
    from exact_attention_85_gb300.inputs import WORKLOADS

    w = WORKLOADS["bf16_b4_h16_n8k_d128_causal"]
    # causal: row r sees r + 1 keys, so N (N + 1) / 2 pairs per head
    assert bench._visible_pairs(w) == 4 * 16 * 8192 * 8193 / 2
    # the metric's convention: 4 B H N^2 d, halved for causal; backward 2.5x
    assert w.fwd_flops() == pytest.approx(4 * 4 * 16 * 8192 ** 2 * 128 / 2)
    assert w.bwd_flops() == pytest.approx(2.5 * w.fwd_flops())
    t = WORKLOADS["tiny_fp16_d64_n256"]
    assert not t.causal and bench._visible_pairs(t) == t.B * t.Hq * 256 * 256


def test_clock_summary_reads_throttle_reasons():
    """The clock record of the timed region: median SM clock over loaded
    samples (power above 300 W), the maximum clock, and every throttle reason
    seen active while loaded (nvidia-smi CSV, no units)."""
    import bench

    c = bench.ClockSampler(0)
    c.out = "\n".join([
        "2070, 2070, 120.5, Not Active, Not Active, Not Active, Not Active",   # idle: ignored
        "2070, 2070, 1150.0, Not Active, Not Active, Not Active, Active",
        "1995, 2070, 1390.2, Not Active, Not Active, Not Active, Active",
        "2055, 2070, 1201.0, Not Active, Active, Not Active, Not Active",
        "garbage line",
        "[N/A], 2070, 900, Not Active, Not Active, Not Active, Not Active",
    ])
    s = c.summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 2055.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    c.out = ""
    assert c.summary()["reasons"] == ["unavailable"]


def test_reference_arm_under_two_ranks_prints_once():
    """Launched as two ranks (the multi-GPU form of the command), the
    reference arm runs on rank 0 alone and prints one line; rank 1 exits 0
    without work."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
