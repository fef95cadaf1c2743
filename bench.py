"""Benchmark of one paged-attention layer step on GB300.

Default workload: Llama-3-70B layer-shape decode with a shared prefix (128
sequences, 64 query / 8 KV heads, head_dim 128; every sequence starts with
the same 2,000-token prefix held once in 125 ref-counted blocks, then a
private tail of floor(exp(U[ln 1K, ln 32K])) tokens; block 124 forked by
copy-on-write; bf16 cache; one new token per sequence appended with
reshape_and_cache through a slot mapping).  A step is the whole hot path for
that batch: the cache write of the new tokens, then paged decode attention
(split-KV partitions merged by the log-sum-exp kernel).

Reported metric: achieved HBM GB/s of the step -- algorithmic bytes (every
K/V element of every sequence read once per token, shared prefix blocks
once, Q read, O written, block-table rows and lengths read, new K/V written)
divided by the measured step time -- and microseconds per layer step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

With --gpus N > 1 (launched by torchrun), every rank runs its own batch of the
same recipe (weak scaling, no collective on the data path); the timed region
is bracketed by barriers and the slowest rank's time is used.
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

METRIC = "paged decode attention: achieved HBM GB/s (% of peak) and µs per layer step"
NOMINAL_HBM_GBS = 8000.0                   # GB300 HBM3e, nominal
UNIT = "GB/s"
L2_BYTES = 129 * 1024 * 1024


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _tensor_peak():
    """Sustained dense bf16 tensor throughput (TFLOP/s) for a kernel timed inside
    a long step, measured on this machine; else the fallback figure."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["bf16_tflops_sustained"]), "measured (sustained)"
    except Exception:
        return 1700.0, "fallback (sustained)"


def prefill_flops(wl):
    """Flops of the chunk rows: 4 * Hq * D per visible key (QK^T and PV)."""
    total = 0
    for L, n in zip(wl.context_lens, wl.q_lens):
        L, n = int(L), int(n)
        if n >= 2:
            total += n * (L - n) + n * (n + 1) // 2
    return 4 * wl.num_q_heads * wl.head_dim * total


def _blocks(n, bs=16):
    return -(-int(n) // bs)


def algorithmic_bytes(wl) -> dict:
    """HBM bytes one step must move at least.

    * ``kv_unique``: every cached K/V element read once per (sequence, KV head),
      counted per token (L tokens x Hkv x D x element bytes, K and V), with the
      tokens of shared prefix blocks counted once.  This is the method's own
      byte count.
    * ``kv_tiles``: the same in whole 16-token (block, head) tiles, which is
      what a block-granular kernel reads: a sequence's last block is fetched
      whole although only L mod 16 of its rows are used.
    * Q read, O written, block-table rows and lengths read, new K/V written."""
    eb = wl.kv_elem_bytes
    tok = 2 * wl.num_kv_heads * wl.head_dim * eb                  # K + V bytes of one token
    tile = wl.block_size * wl.head_dim * eb                       # one (block, head) tile
    nblk = [_blocks(int(L)) for L in wl.context_lens]
    pb = _blocks(wl.prefix_tokens) if wl.prefix_tokens else 0
    # tokens of the prefix blocks every sequence still shares (the copy-on-write
    # block has one private copy per sequence)
    shared_tok = sum(min(16, wl.prefix_tokens - 16 * b) for b in range(pb) if b != wl.cow_block)
    shared_blk = pb - (1 if 0 <= wl.cow_block < pb else 0)
    dupes = max(wl.num_seqs - 1, 0)
    kv_unique = tok * (int(wl.context_lens.sum()) - dupes * shared_tok)
    kv_tiles = 2 * tile * wl.num_kv_heads * (sum(nblk) - dupes * shared_blk)
    kv_logical = tok * int(wl.context_lens.sum())
    q = wl.total_q * wl.num_q_heads * wl.head_dim * 2
    o = wl.total_q * wl.num_q_heads * wl.head_dim * 4
    meta = 4 * sum(nblk) + 4 * wl.num_seqs
    new_kv = 2 * wl.total_q * wl.num_kv_heads * wl.head_dim * (2 + eb) + 8 * wl.total_q
    return {"kv_unique": kv_unique, "kv_tiles": kv_tiles, "kv_logical": kv_logical, "q": q, "o": o,
            "meta": meta, "new_kv": new_kv, "total": kv_unique + q + o + meta + new_kv}


def bench_config(wl, ws, placement) -> dict:
    """The ``config`` object of the JSON line; both arms print the same one."""
    ab = algorithmic_bytes(wl)
    kv_bytes = ab["kv_unique"]
    flush = kv_bytes < 2 * L2_BYTES
    return {"workload": wl.name, "num_seqs": wl.num_seqs, "num_q_heads": wl.num_q_heads,
            "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim, "block_size": wl.block_size,
            "kv_dtype": wl.kv_dtype, "num_blocks": wl.num_blocks,
            "context_tokens": int(wl.context_lens.sum()), "new_tokens_per_step": wl.total_q,
            "prefix_tokens": wl.prefix_tokens,
            "kv_bytes_per_step": kv_bytes, "algorithmic_bytes_per_step": ab["total"],
            "l2": (f"flushed before every timed step ({2 * L2_BYTES / 1e6:.0f} MB written): the "
                   f"{kv_bytes / 1e6:.1f} MB of KV fit in the 129 MB L2") if flush else
                  (f"no flush: every step reads {kv_bytes / 1e6:.0f} MB of KV, "
                   f"{kv_bytes / L2_BYTES:.1f}x the 129 MB L2"),
            "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
            "placement": placement}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, device=None) -> float:
    """Largest value of x across the ranks of the default process group (the
    timing rule: the slowest rank's time); x itself when not distributed."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(bytes_per_rank_step: float, world_size: int, ms_per_step: float) -> float:
    """Whole-job GB/s: every rank processes its own batch of the same size, so
    the units of all ranks are divided by the slowest rank's step time."""
    return world_size * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons while the GPU runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.skip = 0
        self.path = os.path.join("/tmp", f"pkv_clocks_{os.getpid()}.csv")

    def start(self, wait_s=5.0):
        """Start sampling every 100 ms; return once the first sample is written
        (taken before the load starts, so it is left out of the summary)."""
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        t0 = time.monotonic()
        while time.monotonic() - t0 < wait_s and self.proc.poll() is None:
            with open(self.path) as f:
                n = sum(1 for _ in f)
            if n:
                self.skip = n
                return
            time.sleep(0.02)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            lines = f.readlines()[self.skip:]
            for ln in lines:
                p = [x.strip() for x in ln.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    mx.append(float(p[2]))
                except ValueError:
                    continue
                for n, v in zip(names, p[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.remove(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def kernel_source_hash(path):
    """sha256 of the device-code region of a kernel source file (between its
    "device code begin" and "device code end" marker lines)."""
    text = open(path).read()
    a = text.index("// ---- device code begin")
    b = text.index("// ---- device code end")
    return hashlib.sha256(text[a:b].encode()).hexdigest()


def _traffic(kernel_src, workload):
    """Per-launch DRAM bytes of the decode kernel on this workload from the
    committed ncu summary ``profiles/decode_<workload>_traffic.txt``, if that
    summary was taken on the current device code; else None."""
    try:
        kv = {}
        with open(os.path.join(ROOT, "profiles", f"decode_{workload}_traffic.txt")) as f:
            for ln in f:
                if ":" in ln and not ln.startswith("#"):
                    k, v = ln.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_source_sha256") != kernel_source_hash(kernel_src):
            return None
        return int(kv["traffic_bytes_per_launch"])
    except Exception:
        return None


# -------------------------------------------------------------- CPU oracle
class OracleSample:
    """The fp64 oracle (as it stands) on the first ``m`` sequences of the
    workload: block tables from the oracle's allocator model, a compact pool
    holding only those sequences' blocks, the oracle's own scatter; ``run()``
    is one call of the paged oracle on that sample.

    A chunk longer than ``row_cap`` rows is run on its last ``row_cap`` rows
    only.  Its other rows would cost the same per (row, visible key) pair, so
    ``scale`` = (row, key) pairs of the full sample / pairs run, and a call's
    time x ``scale`` estimates the full sample's; ``algo_bytes`` counts the full
    sample."""

    def __init__(self, wl, m, row_cap=16):
        import numpy as np
        import torch

        import oracle
        from oracle import model as omodel
        from synth.workloads import Workload

        self.oracle = oracle
        # every core this process may run on (a launcher's OMP_NUM_THREADS=1 is for
        # its GPU ranks; only one rank runs the oracle)
        self.threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
        m = max(1, min(int(m), wl.num_seqs))
        full_q = np.asarray(wl.q_lens[:m], np.int64)
        run_q = np.minimum(full_q, row_cap) if row_cap else full_q
        lens = np.asarray(wl.context_lens[:m], np.int64)
        self.scale = float((full_q * lens).sum()) / max(1.0, float((run_q * lens).sum()))
        self.capped = bool((run_q < full_q).any())
        sub = Workload(wl.name + "_sample", wl.seed, wl.num_q_heads, wl.num_kv_heads, 0, wl.kv_dtype,
                       wl.context_lens[:m], run_q.astype(np.int32), np.zeros(0, np.int32), wl.prefix_tokens,
                       wl.cow_block, wl.num_splits)
        nblk = int(sum(-(-int(L) // 16) for L in sub.context_lens))
        sub.num_blocks = nblk + (m if sub.cow_block >= 0 else 0)
        sub.free_order = np.arange(sub.num_blocks, dtype=np.int32)
        if sub.kv_dtype == "fp8":
            # the workload's own scales when the GPU arm already scanned them; the
            # reference arm scans the sample's values on the host cores
            if wl._fp8_scales is not None:
                sub._fp8_scales = wl._fp8_scales
            else:
                sub.fp8_scales(device="cpu")
        self.tb = omodel.build_tables(sub)
        self.kc, self.vc = omodel.build_cache(sub, self.tb)
        self.q = sub.q_values().contiguous().view(torch.int16).numpy().view(np.uint16)
        self.code = oracle.FP8 if sub.kv_dtype == "fp8" else oracle.BF16
        self.ks, self.vs = sub.fp8_scales() if self.code == oracle.FP8 else (None, None)
        self.cu = None if sub.is_decode else sub.cu_q_lens
        self.sub, self.m, self.wl = sub, m, wl
        # the bench's own byte count (per token, shared prefix blocks once) for
        # the sample, with Q and O of every row of the full sample
        self.algo_bytes = algorithmic_bytes(sub)["kv_unique"] + int(full_q.sum()) * sub.num_q_heads * 128 * (2 + 4)

    def run(self, nthreads=None):
        self.oracle.paged_attention(self.q, self.kc, self.vc, self.tb.tables, self.sub.context_lens, self.cu,
                                    dtype=self.code, k_scale=self.ks, v_scale=self.vs, scale=self.sub.scale,
                                    nthreads=self.threads if nthreads is None else nthreads)

    def describe(self):
        d = (f"first {self.m} of {self.wl.num_seqs} sequences ({int(self.sub.context_lens.sum())} "
             f"context tokens) of the same workload, fp64 paged oracle")
        if self.capped:
            d += (f"; chunks run on their last {int(self.sub.q_lens.max())} rows, time scaled by "
                  f"{self.scale:.1f} (row, key) pairs of the full sample per pair run")
        return d


def cpu_oracle_baseline(wl, budget_s=10.0, max_seqs=16, single_core=False):
    smp = OracleSample(wl, max_seqs)
    cores = smp.threads

    def timed(nthreads, budget):
        reps, t0 = 0, time.perf_counter()
        while True:
            smp.run(nthreads)
            reps += 1
            el = time.perf_counter() - t0
            if el >= budget:
                return reps, el

    reps, el = timed(cores, budget_s)
    per = el / reps * smp.scale
    out = {"value": smp.algo_bytes / per / 1e9, "unit": UNIT, "cores": cores,
           "kind": "oracle", "sample": f"{smp.describe()}, {reps} calls in {el:.1f} s"}
    if single_core:
        # the same sample on one host core, then the thread count is restored
        r1, e1 = timed(1, budget_s / 2)
        smp.run(cores)
        out["single_core"] = {"value": smp.algo_bytes / (e1 / r1 * smp.scale) / 1e9, "unit": UNIT,
                              "cores": 1, "sample": f"{r1} calls in {e1:.1f} s"}
    return out


def run_reference(args):
    """The oracle as the reference arm: each step is one oracle call on a sample
    of the workload sized so that W + K steps take about two minutes."""
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    from synth.workloads import make_workload
    wl = make_workload(args.workload)
    probe = OracleSample(wl, 1)
    t0 = time.perf_counter()
    probe.run()
    per_seq = max(time.perf_counter() - t0, 1e-6)      # one sequence, chunk rows capped
    budget = args.ref_budget / max(1, args.steps + args.warmup)
    smp = OracleSample(wl, min(args.ref_seqs, max(1, int(budget / per_seq))))
    for _ in range(args.warmup):
        smp.run()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        smp.run()
        times.append(time.perf_counter() - t0)
    total = sum(times) * smp.scale            # the full sample's time (chunk rows capped: scaled)
    v = smp.algo_bytes * len(times) / total / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": bench_config(wl, ws, args.placement),
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": smp.threads, "kind": "oracle",
                             "sample": smp.describe(), "device": "host cores", "time_scale": smp.scale},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def _launches_per_step(pkv, wl):
    """Kernels one step launches: the cache write, then the attention call's
    kernels as the library itself plans them for these sizes (decode + its
    optional LSE merge; for a batch with chunks also the tile-count prefix,
    the chunk kernel and its optional merge)."""
    return 1 + pkv.paged_attention_launch_count(wl.num_seqs, int(wl.q_lens.sum()), int(wl.q_lens.max()), wl.num_q_heads, wl.num_kv_heads,
                                                wl.max_blocks_per_seq, wl.num_splits)


# ------------------------------------------------------------------ ours
def _e2e_pipelined(dw, parts, offs, d_pack, h_pack, stream, dev, E, barrier, max_over_ranks):
    """End-to-end steps overlapped the way a serving loop runs them: step i's
    packed inputs go up on one copy stream and its output comes down on
    another, into and out of one of two buffer sets, while the compute stream
    runs the neighbouring steps.  Returns ms per step over E steps."""
    import torch

    sets = []
    for _ in range(2):
        dp = torch.empty_like(d_pack)
        views = {}
        for (name, t), o in zip(parts, offs):
            n = t.numel() * t.element_size()
            views[name] = dp[o:o + n].view(t.dtype).view(t.shape)
        op = torch.empty_like(dw.out)
        ho = torch.empty(op.shape, dtype=op.dtype).pin_memory()
        sets.append((dp, views, op, ho))
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    freed = [torch.cuda.Event() for _ in range(2)]
    keep = {name: getattr(dw, name) for name, _ in parts}
    keep_out = dw.out

    def run(n, start):
        up.wait_event(start)
        for i in range(n):
            b = i % 2
            dp, views, op, ho = sets[b]
            with torch.cuda.stream(up):
                if i >= 2:
                    up.wait_event(freed[b])        # step i-2 computed and read back
                dp.copy_(h_pack, non_blocking=True)
                ready[b].record(up)
            stream.wait_event(ready[b])
            for name, v in views.items():
                setattr(dw, name, v)
            dw.out = op
            dw.step()
            done[b].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(done[b])
                ho.copy_(op, non_blocking=True)
                freed[b].record(down)
        stream.wait_stream(down)
        stream.wait_stream(up)

    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run(3, e0)
    barrier()
    e0.record(stream)
    run(E, e0)
    e1.record(stream)
    barrier()
    ms = max_over_ranks(e0.elapsed_time(e1) / E, dev)
    for name, v in keep.items():
        setattr(dw, name, v)
    dw.out = keep_out
    return ms


def run_ours(args):
    import torch

    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import paged_kv_cache_263_gb300 as pkv
    from paged_kv_cache_263_gb300 import build as pkv_build
    from paged_kv_cache_263_gb300.workload import DeviceWorkload
    from synth.workloads import make_workload

    pkv_build.build()
    wl = make_workload(args.workload)
    if args.placement == "contiguous":
        # the paged-vs-contiguous comparison: the pool hands out blocks in
        # ascending order, so every sequence's blocks are consecutive in HBM
        import numpy as np
        wl.free_order = np.arange(wl.num_blocks, dtype=np.int32)
    dw = DeviceWorkload(wl, device=dev)
    ab = algorithmic_bytes(wl)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    dw.step()
    st = pkv.kv_last_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} flags {pkv.kv_last_device_status_flags()}")

    # ---- device-resident timed region.  The step is captured once into a CUDA
    # graph (cache write + attention, every kernel of the step) and replayed: a
    # layer step is launch-bound when the batch is small, and graph replay is
    # how the step runs on the GPU without per-launch host overhead.  A second
    # graph holds the attention call alone, for the roofline's per-call time.
    K = args.steps
    graphs = None
    try:
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for _ in range(3):
                dw.step()
        stream.wait_stream(side)
        torch.cuda.synchronize(dev)
        g_step, g_attn = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_step):
            dw.write_new_tokens()
            dw.attention()
        with torch.cuda.graph(g_attn):
            dw.attention()
        torch.cuda.synchronize(dev)
        graphs = (g_step, g_attn)
    except Exception as e:                  # capture refused: eager timing only
        graph_error = f"{type(e).__name__}: {e}"[:200]
        torch.cuda.synchronize(dev)
    clocks = Clocks(local)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    # a workload whose K/V fits in L2 is timed step by step with L2 flushed
    # (a 2x-L2 buffer overwritten, outside the timed events) before each step
    flush = ab["kv_unique"] < 2 * L2_BYTES
    flush_buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev) if flush else None

    def clock_window(one_step):
        """Sample the clocks under load: nvidia-smi starts, then the step runs
        back to back for at least --clock-window seconds right before the timed
        region (untimed), and the sampler keeps running through the timed
        steps.  A timed region of a few ms alone would see no sample."""
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(3):
            one_step()
        b.record(stream)
        torch.cuda.synchronize(dev)
        est_ms = max(a.elapsed_time(b) / 3, 1e-3)
        n = max(1, int(args.clock_window * 1e3 / est_ms) + 1)
        clocks.start()
        for i in range(n):
            one_step()
            if i % 256 == 255:
                torch.cuda.synchronize(dev)    # keep the host from running far ahead
        barrier()
        return n

    if graphs:
        g_step, g_attn = graphs
        for _ in range(args.warmup):
            if flush:
                flush_buf.zero_()
            g_step.replay()
        barrier()
        if flush:
            def one():
                flush_buf.zero_()
                g_step.replay()
            window_steps = clock_window(one)
            fe = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
            t_start.record(stream)
            for i in range(K):
                flush_buf.zero_()
                fe[i][0].record(stream)
                g_step.replay()
                fe[i][1].record(stream)
            t_end.record(stream)
            barrier()
            ck = clocks.stop()
            ms_per_step = max_over_ranks(sum(a.elapsed_time(b) for a, b in fe) / K, dev)
            fa = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
            for i in range(K):
                flush_buf.zero_()
                fa[i][0].record(stream)
                g_attn.replay()
                fa[i][1].record(stream)
            torch.cuda.synchronize(dev)
            attn_avg_graph = sum(a.elapsed_time(b) for a, b in fa) / K
        else:
            window_steps = clock_window(g_step.replay)
            t_start.record(stream)
            for i in range(K):
                g_step.replay()
            t_end.record(stream)
            barrier()
            ck = clocks.stop()
            total_ms = max_over_ranks(t_start.elapsed_time(t_end), dev)
            ms_per_step = total_ms / K
            # attention alone, same graph mechanism
            for _ in range(3):
                g_attn.replay()
            torch.cuda.synchronize(dev)
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            for _ in range(K):
                g_attn.replay()
            a1.record(stream)
            torch.cuda.synchronize(dev)
            attn_avg_graph = a0.elapsed_time(a1) / K
        st = pkv.kv_last_device_status()
        if st != 0:
            raise RuntimeError(f"device status {st} after the graph replays "
                               f"(flags {pkv.kv_last_device_status_flags()})")
    # eager: the same step issued call by call (host launch overhead included),
    # with events around each call
    KE = min(K, 1000)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(KE)]
    for _ in range(args.warmup):
        dw.step()
    barrier()
    if not graphs:
        window_steps = clock_window(dw.step)
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    for i in range(KE):
        ev[i][0].record(stream)
        dw.write_new_tokens()
        ev[i][1].record(stream)
        dw.attention()
        ev[i][2].record(stream)
    e_end.record(stream)
    barrier()
    eager_ms = max_over_ranks(e_start.elapsed_time(e_end), dev) / KE
    attn_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(KE)]
    write_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(KE)]
    if not graphs:
        ck = clocks.stop()
        ms_per_step = eager_ms
    st = pkv.kv_last_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} after timing (flags {pkv.kv_last_device_status_flags()})")

    # ---- end to end through the public API with pinned host buffers.  A step's
    # inputs (queries, new K/V, slots, block tables, lengths) sit packed in one
    # pinned host buffer and move with one host->device copy into one device
    # buffer whose views the calls take; the output comes back with one copy.
    parts = [("q", dw.q), ("new_k", dw.new_k), ("new_v", dw.new_v), ("slot_mapping", dw.slot_mapping),
             ("block_tables", dw.block_tables), ("context_lens", dw.context_lens)]
    if not wl.is_decode:
        parts.append(("cu_q_lens", dw.cu_q_lens))
    offs, packed = [], 0
    for _, t in parts:
        offs.append(packed)
        packed += (t.numel() * t.element_size() + 255) // 256 * 256
    d_pack = torch.empty(packed, dtype=torch.uint8, device=dev)
    h_pack = torch.empty(packed, dtype=torch.uint8).pin_memory()
    for (name, t), o in zip(parts, offs):
        n = t.numel() * t.element_size()
        h_pack[o:o + n].view(t.dtype).view(t.shape).copy_(t.cpu())
        setattr(dw, name, d_pack[o:o + n].view(t.dtype).view(t.shape))
    h_out = torch.empty(dw.out.shape, dtype=torch.float32).pin_memory()
    h2d = packed
    d2h = h_out.numel() * h_out.element_size()
    E = max(3, min(K, 200))

    def e2e_step():
        d_pack.copy_(h_pack, non_blocking=True)
        dw.step()
        h_out.copy_(dw.out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(E):
        e2e_step()
    e1.record(stream)
    barrier()
    e2e_eager_ms = max_over_ranks(e0.elapsed_time(e1) / E, dev)
    # the same end-to-end step (host->device inputs, cache write, attention,
    # device->host output) captured once and replayed, as a serving loop runs it
    e2e_ms, e2e_kind = e2e_eager_ms, "eager calls"
    if graphs:
        try:
            g_e2e = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_e2e):
                e2e_step()
            for _ in range(3):
                g_e2e.replay()
            barrier()
            e0.record(stream)
            for _ in range(E):
                g_e2e.replay()
            e1.record(stream)
            barrier()
            e2e_ms, e2e_kind = max_over_ranks(e0.elapsed_time(e1) / E, dev), "CUDA graph replay of the whole step"
        except Exception:
            torch.cuda.synchronize(dev)
    pipe_ms = _e2e_pipelined(dw, parts, offs, d_pack, h_pack, stream, dev, E, barrier, max_over_ranks)

    peak, peak_kind = _peaks()
    step_bytes = ab["total"]
    value = weak_scaling_value(step_bytes, ws, ms_per_step)
    attn_bytes = ab["kv_unique"] + ab["q"] + ab["o"] + ab["meta"]
    attn_avg = attn_avg_graph if graphs else statistics.mean(attn_ms)
    hpeak, _ = _peaks()
    tpeak, tkind = _tensor_peak()
    # memory-bound unless the chunk rows' flops per byte reach the ridge point
    hbm_bound = wl.is_decode or prefill_flops(wl) / attn_bytes < tpeak * 1e12 / (hpeak * 1e9)
    if hbm_bound:
        achieved = attn_bytes / (attn_avg * 1e-3) / 1e9
        roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                    "frac": achieved / peak, "peak_kind": peak_kind,
                    "kernel": "paged_attention_decode (decode kernel + LSE reduce)" if wl.is_decode else
                              "paged_attention_chunked_prefill (whole call)",
                    "bytes_per_launch": attn_bytes, "avg_launch_ms": attn_avg,
                    "bytes": "K/V per token (L x Hkv x 128 x 2 tensors x element bytes, shared prefix "
                             "blocks once) + Q + O + block-table rows and lengths",
                    "kv_tile_bytes_per_launch": ab["kv_tiles"],
                    "traffic": _traffic(os.path.join(ROOT, "paged_kv_cache_263_gb300", "csrc", "decode.cu"),
                                        wl.name) if wl.is_decode else None}
    else:
        flops = prefill_flops(wl)
        # the chunk kernel's own launches, timed with the library's trace events
        # on the launching stream (eager calls after the timed region)
        pkv.kv_trace_prefill(True)
        kern_ms = []
        for _ in range(max(3, min(K, 20))):
            dw.attention()
            t = pkv.kv_trace_prefill_kernel_ms()
            if t > 0:
                kern_ms.append(t)
        pkv.kv_trace_prefill(False)
        kern_avg = statistics.mean(kern_ms) if kern_ms else attn_avg
        achieved = flops / (kern_avg * 1e-3) / 1e12
        call_tflops = flops / (attn_avg * 1e-3) / 1e12
        roofline = {"bound": "tensor", "achieved": achieved, "peak": tpeak, "unit": "TFLOP/s",
                    "frac": achieved / tpeak, "peak_kind": tkind,
                    "kernel": ("prefill_kernel (tcgen05 chunk tiles), its own launches" if kern_ms else
                               "paged_attention_chunked_prefill (whole call)"),
                    "flops_per_launch": flops, "avg_launch_ms": kern_avg, "traffic": None,
                    "whole_call": {"avg_ms": attn_avg, "achieved": call_tflops, "frac": call_tflops / tpeak,
                                   "includes": "chunk tiles + decode rows (beside them) + LSE merges"}}
    launches_per_step = _launches_per_step(pkv, wl)
    kv_bytes = ab["kv_unique"]
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "us_per_layer_step": ms_per_step * 1e3,
        "pct_of_peak": 100.0 * value / ws / peak,
        # against the ~8 TB/s nominal HBM3e bandwidth that the target is stated in
        "pct_of_nominal_peak": 100.0 * value / ws / NOMINAL_HBM_GBS,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if wl.kv_dtype == "bf16" else "fp8-e4m3 cache, f16 math",
        "data": "synthetic",
        "config": bench_config(wl, ws, args.placement),
        "roofline": roofline,
        "cache_write_avg_ms": statistics.mean(write_ms),
        "timing": ("CUDA graph replay of the captured step (cache write + attention); roofline per call "
                   "from a graph of the attention call alone") if graphs else
                  f"eager calls (graph capture failed: {graph_error})",
        "eager": {"ms_per_step": eager_ms, "attention_call_ms": statistics.mean(attn_ms), "steps": KE},
        "e2e": {"value": weak_scaling_value(step_bytes, ws, e2e_eager_ms), "unit": UNIT,
                "ms_per_step": e2e_eager_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "timing": "eager calls of the public API, copies included",
                "graph": {"value": weak_scaling_value(step_bytes, ws, e2e_ms), "ms_per_step": e2e_ms,
                          "timing": e2e_kind},
                "pipelined": {"value": weak_scaling_value(step_bytes, ws, pipe_ms), "ms_per_step": pipe_ms,
                              "timing": "eager calls as a serving loop overlaps them: two sets of input and "
                                        "output buffers, step i+1's inputs up and step i-1's output down on "
                                        "copy streams while step i computes; every step moves its own bytes"}},
        "gpu_launches": launches_per_step * K,
        "clocks": ck,
        "clock_window": {"steps": window_steps, "seconds_min": args.clock_window,
                         "timing": "untimed back-to-back steps right before the timed region, sampled "
                                   "with nvidia-smi every 100 ms together with the timed steps"},
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_baseline(wl, budget_s=args.cpu_budget, single_core=wl.name == "tiny")
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------------------ swap
SWAP_METRIC = "KV block swap over the host link: GB/s moved (swap-out + swap-in of 1.07 GB)"


def _link_peaks(torch, dev, nbytes, reps=5):
    """Measured copy-engine bandwidth of one contiguous pinned host <-> device
    copy of nbytes each way (best of reps), in GB/s."""
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    s = torch.cuda.current_stream(dev)
    out = {}
    for name, fn in (("d2h", lambda: h.copy_(d, non_blocking=True)), ("h2d", lambda: d.copy_(h, non_blocking=True))):
        best = None
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            fn()
            b.record(s)
            torch.cuda.synchronize(dev)
            ms = a.elapsed_time(b)
            best = ms if best is None else min(best, ms)
        out[name] = nbytes / (best * 1e-3) / 1e9
    del h, d
    return out


def run_swap(args):
    """One step = swap-out of 16,384 (block, all 8 KV heads) bf16 blocks of K and
    V (1.07 GB, the page's preempted request) from a 32,768-block pool to pinned
    host memory, then swap-in of the same bytes into 16,384 other blocks."""
    import numpy as np
    import torch

    import paged_kv_cache_263_gb300 as pkv
    from paged_kv_cache_263_gb300 import build as pkv_build

    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pkv_build.build()
    NB, HKV, N = 32768, 8, 16384
    rng = np.random.Generator(np.random.PCG64(2636 + rank))
    perm = rng.permutation(NB).astype(np.int32)
    out_ids = torch.from_numpy(perm[:N].copy()).to(dev)
    in_ids = torch.from_numpy(perm[N:].copy()).to(dev)
    k = torch.empty((NB, HKV, 16, 128), dtype=torch.bfloat16, device=dev).normal_()
    v = torch.empty_like(k).normal_()
    hk = torch.empty((N, HKV, 16, 128), dtype=torch.bfloat16).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    moved = 2 * N * HKV * 16 * 128 * 2                       # bytes of one direction (K + V)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    # correctness of the timed configuration before timing: a sample of blocks
    pkv.kv_swap_out(k, v, out_ids, hk, hv)
    pkv.kv_swap_in(k, v, in_ids, hk, hv)
    torch.cuda.synchronize(dev)
    if pkv.kv_last_device_status() != 0:
        raise RuntimeError("device status after swap")
    for j in (0, 1, N // 2, N - 1):
        a, b = int(perm[j]), int(perm[N + j])
        if not (torch.equal(k[a], k[b]) and torch.equal(v[a], v[b]) and torch.equal(hk[j], k[a].cpu())):
            raise RuntimeError(f"swap mismatch at {j}")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    clocks = Clocks(local)
    clocks.start()
    for _ in range(args.warmup):
        pkv.kv_swap_out(k, v, out_ids, hk, hv)
        pkv.kv_swap_in(k, v, in_ids, hk, hv)
    barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(K):
        ev[i][0].record(stream)
        pkv.kv_swap_out(k, v, out_ids, hk, hv)
        ev[i][1].record(stream)
        pkv.kv_swap_in(k, v, in_ids, hk, hv)
        ev[i][2].record(stream)
    t1.record(stream)
    barrier()
    ck = clocks.stop()
    ms_step = max_over_ranks(t0.elapsed_time(t1) / K, dev)
    out_ms = statistics.mean(ev[i][0].elapsed_time(ev[i][1]) for i in range(K))
    in_ms = statistics.mean(ev[i][1].elapsed_time(ev[i][2]) for i in range(K))

    # end to end: the block ids come from the host scheduler each step
    h_out = torch.from_numpy(perm[:N].copy()).pin_memory()
    h_in = torch.from_numpy(perm[N:].copy()).pin_memory()
    E = max(3, min(K, 20))
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(E):
        out_ids.copy_(h_out, non_blocking=True)
        in_ids.copy_(h_in, non_blocking=True)
        pkv.kv_swap_out(k, v, out_ids, hk, hv)
        pkv.kv_swap_in(k, v, in_ids, hk, hv)
    e1.record(stream)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / E, dev)

    link = _link_peaks(torch, dev, moved)
    out_gbs = moved / (out_ms * 1e-3) / 1e9
    in_gbs = moved / (in_ms * 1e-3) / 1e9
    peak = min(link["d2h"], link["h2d"])
    achieved = 2 * moved / ((out_ms + in_ms) * 1e-3) / 1e9
    line = {
        "metric": SWAP_METRIC, "value": weak_scaling_value(2 * moved, ws, ms_step), "unit": "GB/s",
        "n_gpus": ws, "steps": K, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16 (bytes moved)",
        "data": "synthetic",
        "config": {"workload": "swap", "pool_blocks": NB, "num_kv_heads": HKV, "blocks_per_direction": N,
                   "bytes_per_direction": moved, "host_memory": "pinned (cudaHostAlloc via torch)",
                   "l2": "no flush: 1.07 GB each way, 8x the 129 MB L2",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "swap_out": {"ms": out_ms, "GB/s": out_gbs}, "swap_in": {"ms": in_ms, "GB/s": in_gbs},
        "roofline": {"bound": "host link", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": "measured live: one contiguous pinned copy of "
                     "the same bytes each way by the copy engine (d2h %.1f, h2d %.1f GB/s); lower of the two"
                     % (link["d2h"], link["h2d"]),
                     "kernel": "swap_kernel (out and in)", "bytes_per_launch": moved,
                     "avg_launch_ms": (out_ms + in_ms) / 2, "traffic": None},
        "e2e": {"value": weak_scaling_value(2 * moved, ws, e2e_ms), "unit": "GB/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": moved + 2 * N * 4, "d2h_bytes_per_step": moved},
        "gpu_launches": 2 * K,
        "clocks": ck,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = _swap_cpu_baseline(args.cpu_budget)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def _swap_cpu_baseline(budget_s):
    """The swap oracle (numpy gather of the listed blocks, then scatter into
    others) on host arrays: 2,048 of the 16,384 blocks, 134 MB each way."""
    import numpy as np
    from oracle.swap import swap_in as o_in, swap_out as o_out
    rng = np.random.Generator(np.random.PCG64(2636))
    NB, HKV, N = 4096, 8, 2048
    k = rng.integers(0, 1 << 16, size=(NB, HKV, 16, 128), dtype=np.uint16)
    v = rng.integers(0, 1 << 16, size=(NB, HKV, 16, 128), dtype=np.uint16)
    perm = rng.permutation(NB)
    reps, t0 = 0, time.perf_counter()
    while True:
        hk, hv = o_out(k, v, perm[:N])
        o_in(k, v, perm[N:], hk, hv)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    moved = 2 * 2 * N * HKV * 16 * 128 * 2
    return {"value": moved * reps / el / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{N} of 16,384 blocks each way (numpy gather/scatter), {reps} round trips in {el:.1f} s"}


def run_swap_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    steps = []
    for _ in range(args.warmup):
        _swap_cpu_baseline(0.0)
    for _ in range(args.steps):
        steps.append(_swap_cpu_baseline(0.0))
    v = statistics.mean(s["value"] for s in steps)
    line = {"impl": "reference", "metric": SWAP_METRIC, "value": v, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": None, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bytes", "data": "synthetic",
            "config": {"workload": "swap", "sample": steps[0]["sample"], "device": "host cores"},
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": steps[0]["sample"]},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=500)
    ap.add_argument("--workload", default="llama70b_prefix")
    ap.add_argument("--clock-window", type=float, default=1.0,
                    help="seconds of untimed steps, sampled for clocks, right before the timed region")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--ref-seqs", type=int, default=16)
    ap.add_argument("--ref-budget", type=float, default=120.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--placement", default="random", choices=["random", "contiguous"],
                    help="physical block placement: the workload's seeded random order, or ascending "
                         "(each sequence's blocks consecutive) for the paged-vs-contiguous comparison")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.workload == "swap":
        return run_swap_reference(args) if args.impl == "reference" else run_swap(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
