"""The benchmark's output contract, checked on the CPU: `bench.py --impl
reference` (the oracle timed on the host cores) prints one JSON line with the
keys and types the contract fixes. The GPU arm's line is produced by the same
report code; its keys are checked here against a line built from fake
timings."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

BASE_KEYS = {"metric": str, "value": (int, float), "unit": str, "n_gpus": int, "steps": int,
             "warmup": int, "ms_per_step": (int, float), "higher_is_better": bool,
             "scaling": str, "dtype": str, "data": str, "config": dict}


def _check_base(line):
    for k, t in BASE_KEYS.items():
        assert k in line, k
        assert isinstance(line[k], t), (k, type(line[k]))
    assert "vs_baseline" in line and line["vs_baseline"] is None
    assert line["config"]["workload"]
    assert line["warmup"] >= 3


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "2", "--warmup", "1",
                        "--cpu-tokens", "64"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.strip().splitlines() if l.strip()]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    _check_base(line)
    assert line["impl"] == "reference"
    assert line["gpu_launches"] == 0
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"]
    assert cb["value"] == line["value"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_gpu_arm_report_has_the_contract_keys():
    torch = pytest.importorskip("torch")
    del torch
    import argparse
    import bench
    import workloads as W

    w = W.get("large_expert")
    args = argparse.Namespace(steps=100, warmup=5, fp8=False, gumbel=None, no_cpu=True,
                              cpu_tokens=64)
    stage = [0.075, 0.014, 0.12, 4.8, 4.6, 0.11]
    clk = {"sm_mhz": 1780.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 5}
    e2e = {"ms": 10.0, "h2d": w.T * w.H * 2, "d2h": w.T * w.H * 2 + 4}
    m = {"ms": sum(stage), "stage_ms": stage, "status": 0, "n_kept": 65536, "any_kept": 32768,
         "l2": "inputs larger than L2", "steps": 100, "host_window": (0.0, 1.0)}
    line = bench.report(args, w, 1, m, clk, e2e, None, dense=4.6)
    _check_base(line)
    rf = line["roofline"]
    assert rf["bound"] == "tensor" and rf["unit"] == "TFLOP/s"
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    # the timed region is well under a second: the burst peak is the roofline
    assert rf["peak"] == bench.peaks()["bf16_tflops"]
    # achieved = the GEMMs' algorithmic FLOP over their event time
    flop = 4 * 65536 * w.H * w.h
    assert abs(rf["achieved"] - flop / (9.4e-3) / 1e12) < 1.0
    assert line["e2e"]["h2d_bytes_per_step"] == w.T * w.H * 2
    assert line["gpu_launches"] == 7 * args.steps
    assert line["clocks"]["reasons"] == ["sw_power_cap"]
    assert line["moe_vs_dense_ffn"]["ratio"] == round(sum(stage) / 4.6, 3)
    json.dumps(line)  # serialisable
    # a per-workload entry has the same accounting, FP8 against twice the peak
    kr = bench.kernel_report(w, m, True)
    assert kr["roofline"]["peak"] == 2 * bench.peaks()["bf16_tflops"]
    assert kr["value"] == round(w.T / (sum(stage) / 1e3), 1)


def test_clock_window_keeps_samples_of_the_timed_region_only(tmp_path):
    import bench
    c = bench.ClockSampler(0)
    row = lambda t, mhz, cap: [t, "0", str(mhz), "2070", "900.0", "0x0", "Not Active",
                               "Not Active", "Not Active", cap]
    c.rows = [row(0.9, 2070, "Not Active"), row(1.01, 1500, "Active"),
              row(1.06, 1600, "Active"), row(1.11, 1700, "Not Active"),
              row(1.5, 2070, "Not Active")]
    win = c.window(1.0, 1.1)
    assert win["samples"] == 3 and win["sm_mhz"] == 1600
    assert win["reasons"] == ["sw_power_cap"] and win["sm_max_mhz"] == 2070


def test_reference_arm_under_torchrun_prints_once():
    """Launched with torchrun for N = 2 on 127.0.0.1: rank 0 alone runs the
    oracle and prints the line; the other rank exits 0."""
    import socket
    with socket.socket() as sock:
        sock.bind(("127.0.0.1", 0))
        port = sock.getsockname()[1]
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                        "--nproc-per-node", "2", "--master-addr", "127.0.0.1",
                        "--master-port", str(port), os.path.join(ROOT, "bench.py"),
                        "--impl", "reference", "--gpus", "2", "--workload", "tiny",
                        "--steps", "1", "--warmup", "1", "--cpu-tokens", "32"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.strip().splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    _check_base(line)
    assert line["impl"] == "reference" and line["n_gpus"] == 2
