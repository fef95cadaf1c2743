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
    # both arms print the same config object
    b = _bench_module()
    from synth.workloads import make_workload
    assert d["config"] == b.bench_config(make_workload(workload), 1, "random")
    # a long chunk is sampled on a few rows, its time scaled by (row, key) pairs
    cb = d["cpu_baseline"]
    assert cb["time_scale"] >= 1.0
    if workload == "mixed_prefill_small":
        assert cb["time_scale"] > 10 and "scaled" in cb["sample"]
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
    assert b._traffic(src, "llama8b") == int(recorded["traffic_bytes_per_launch"])
    # the same file with one device-code line changed
    text = open(src).read()
    a = text.index("// ---- device code begin")
    edited = text[:a] + text[a:].replace("griddep_wait();", "griddep_wait(); ", 1)
    p = tmp_path / "decode.cu"
    p.write_text(edited)
    assert b.kernel_source_hash(str(p)) != b.kernel_source_hash(src)
    assert b._traffic(str(p), "llama8b") is None
    assert b._traffic(src, "no_such_workload") is None


def test_launches_per_step_from_the_library_plan():
    """gpu_launches = steps x (cache write + the kernels the library plans for the
    attention call), counted without a GPU."""
    b = _bench_module()
    import paged_kv_cache_263_gb300 as pkv
    from synth.workloads import make_workload
    expect = {"llama8b": 3,          # write, decode, LSE merge
              "tiny": 3,
              "spec_verify": 4,      # write, work list, chunk kernel, chunk merge (no decode rows)
              "mixed_prefill": 6,    # write, decode rows + merge, work list, chunk kernel, chunk merge
              "spec_verify8": 4}
    for name, n in expect.items():
        assert b._launches_per_step(pkv, make_workload(name)) == n, name


def test_algorithmic_bytes_count_tokens_and_the_shared_prefix_once():
    """K/V bytes are per token (L x Hkv x 128 x 2 x element bytes), the shared
    prefix blocks once; whole 16-token tiles are reported beside them."""
    b = _bench_module()
    from synth.workloads import make_workload, small_workload
    wl = make_workload("llama8b")
    ab = b.algorithmic_bytes(wl)
    assert ab["kv_unique"] == int(wl.context_lens.sum()) * 8 * 128 * 2 * 2
    assert ab["kv_tiles"] == sum(-(-int(L) // 16) for L in wl.context_lens) * 8 * 16 * 128 * 2 * 2
    assert ab["kv_tiles"] - ab["kv_unique"] < 64 * 16 * 8 * 128 * 4
    # 70B shape: 124 prefix blocks shared by all 128 sequences, block 124 forked per sequence
    wl = make_workload("llama70b_prefix")
    ab = b.algorithmic_bytes(wl)
    tok = 8 * 128 * 2 * 2
    assert ab["kv_unique"] == tok * (int(wl.context_lens.sum()) - 127 * 1984)
    assert ab["kv_logical"] - ab["kv_unique"] == tok * 127 * 1984
    # a 40-token prefix: blocks 0 and 1 shared (32 tokens), block 2 (8 tokens) forked
    wl = small_workload(5, lens=[50, 60, 70], prefix_tokens=40, cow_block=2, hkv=2)
    ab = b.algorithmic_bytes(wl)
    assert ab["kv_unique"] == 2 * 128 * 2 * 2 * (180 - 2 * 32)
    # fp8: one byte per element
    wl = make_workload("split_fp8")
    assert b.algorithmic_bytes(wl)["kv_unique"] == 8 * 131072 * 8 * 128 * 2
