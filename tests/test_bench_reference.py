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


def _bench_module():
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_for_tests", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    return b


def test_roofline_traffic_only_while_the_profiled_kernel_is_unchanged(tmp_path):
    """roofline.traffic comes from the committed ncu summary only while the hash
    of decode.cu's device-code region matches the one recorded with the counters;
    an edited kernel reports null."""
    b = _bench_module()
    src = os.path.join(ROOT, "paged_kv_cache_263_gb300", "csrc", "decode.cu")
    with open(os.path.join(ROOT, "profiles", "decode_llama8b_traffic.txt")) as f:
        recorded = dict(l.split(":", 1) for l in f if ":" in l and not l.startswith("#"))
    assert b.kernel_source_hash(src) == recorded["kernel_source_sha256"].strip()
    assert b._traffic(src) == int(recorded["traffic_bytes_per_launch"])
    # the same file with one device-code line changed
    text = open(src).read()
    a = text.index("// ---- device code begin")
    edited = text[:a] + text[a:].replace("griddep_wait();", "griddep_wait(); ", 1)
    p = tmp_path / "decode.cu"
    p.write_text(edited)
    assert b.kernel_source_hash(str(p)) != b.kernel_source_hash(src)
    assert b._traffic(str(p)) is None


def test_launches_per_step_from_the_library_plan():
    """gpu_launches = steps x (cache write + the kernels the library plans for the
    attention call), counted without a GPU."""
    b = _bench_module()
    import paged_kv_cache_263_gb300 as pkv
    from synth.workloads import make_workload
    expect = {"llama8b": 3,          # write, decode, LSE merge
              "tiny": 3,
              "spec_verify": 3,      # write, multi-row decode, merge
              "mixed_prefill": 6,    # write, decode rows + merge, tile prefix, chunk kernel, chunk merge
              "spec_verify8": 6}
    for name, n in expect.items():
        assert b._launches_per_step(pkv, make_workload(name)) == n, name
