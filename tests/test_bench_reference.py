"""bench.py's reference arm runs on host cores only (the fp64 oracle), so its
JSON line can be checked here: the keys of the contract, a positive
throughput, and a cpu_baseline describing the same run."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _line(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", *args],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


@pytest.mark.parametrize("workload", ["tiny", "mixed_prefill_small"])
def test_reference_arm_line(workload):
    d = _line("--workload", workload, "--steps", "1", "--warmup", "3", "--ref-seqs", "2", "--ref-budget", "2")
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["config"]["workload"] == workload and d["dtype"] == "f64" and d["data"] == "synthetic"
    # a long chunk is sampled on a few rows, its time scaled by (row, key) pairs
    assert d["config"]["time_scale"] >= 1.0
    if workload == "mixed_prefill_small":
        assert d["config"]["time_scale"] > 10 and "scaled" in d["config"]["sample"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_enforces_three_warmup_steps():
    d = _line("--workload", "tiny", "--steps", "1", "--warmup", "0", "--ref-seqs", "1", "--ref-budget", "1")
    assert d["warmup"] == 3


def test_reference_arm_under_torchrun_two_ranks():
    """Launched as the driver launches N > 1: rank 0 alone runs the oracle and
    prints one line (on every core of its affinity set); the other rank exits 0
    without work."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port),
                        os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--workload", "tiny",
                        "--steps", "1", "--warmup", "3", "--ref-seqs", "1", "--ref-budget", "1"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    affinity = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    assert d["cpu_baseline"]["cores"] == affinity
