"""Replays a synthetic workload through the oracle (test infrastructure only).

Produces, with the oracle's own code only:
  * block tables from the Python block-manager model (LIFO free list,
    refcounted prefix sharing, copy-on-write forks);
  * cache bytes from the oracle's scatter of the generator's K/V rows;
  * fp64 attention outputs, either over the whole paged cache (small
    workloads) or for chosen sequences / query rows straight from the
    generator's contiguous values (any size).

The order of operations is the workload recipe: allocate and write the shared
prefix, let every other sequence share it, fork the copy-on-write block of
each sequence, then allocate and write every sequence's own tokens.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import BF16, FP8, contiguous_attention, e4m3_decode, e4m3_encode, paged_attention
from . import reshape_and_cache as _scatter
from .allocator import PoolModel, blocks_for


@dataclass
class TableBuild:
    tables: np.ndarray          # int32 [B][max_blocks], -1 where unused
    pool: PoolModel
    prefix_ids: list            # physical prefix blocks as first allocated
    copies: list                # (src, dst) block copies made by copy-on-write


def build_tables(wl) -> TableBuild:
    pool = PoolModel(wl.num_blocks, wl.free_order)
    B, mb, bs = wl.num_seqs, wl.max_blocks_per_seq, wl.block_size
    tables = np.full((B, mb), -1, dtype=np.int32)
    pb = blocks_for(wl.prefix_tokens, bs) if wl.prefix_tokens else 0
    prefix_ids = []
    if pb:
        prefix_ids = pool.alloc(pb)
        tables[0, :pb] = prefix_ids
        for s in range(1, B):
            pool.share(prefix_ids)
            tables[s, :pb] = prefix_ids
    copies = []
    if wl.cow_block >= 0:
        for s in range(B):
            old = int(tables[s, wl.cow_block])
            new, need_copy = pool.copy_on_write(old)
            if need_copy:
                copies.append((old, new))
            tables[s, wl.cow_block] = new
    for s in range(B):
        n = blocks_for(int(wl.context_lens[s]), bs) - pb
        ids = pool.alloc(n)
        tables[s, pb:pb + n] = ids
    return TableBuild(tables, pool, prefix_ids, copies)


def slots_for(table_row: np.ndarray, t0: int, t1: int, block_size: int = 16) -> np.ndarray:
    t = np.arange(t0, t1, dtype=np.int64)
    return table_row[t // block_size].astype(np.int64) * block_size + t % block_size


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def build_cache(wl, tb: TableBuild | None = None):
    """Oracle cache arrays (numpy, uint16 bf16 bits or uint8 e4m3) after the
    workload's writes, including the step's new tokens."""
    if tb is None:
        tb = build_tables(wl)
    dt = np.uint8 if wl.kv_dtype == "fp8" else np.uint16
    shape = (wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim)
    kc = np.zeros(shape, dtype=dt)
    vc = np.zeros(shape, dtype=dt)
    code = FP8 if wl.kv_dtype == "fp8" else BF16
    ks, vs = wl.fp8_scales() if code == FP8 else (None, None)
    bs = wl.block_size
    if wl.prefix_tokens:
        row = np.full(wl.max_blocks_per_seq, -1, dtype=np.int32)
        row[:len(tb.prefix_ids)] = tb.prefix_ids
        slots = slots_for(row, 0, wl.prefix_tokens, bs)
        _scatter(_bits(wl.seq_kv("k", 0, 0, wl.prefix_tokens)), _bits(wl.seq_kv("v", 0, 0, wl.prefix_tokens)),
                 kc, vc, slots, code, ks, vs)
    for src, dst in tb.copies:
        kc[dst] = kc[src]
        vc[dst] = vc[src]
    for s in range(wl.num_seqs):
        t0 = wl.prefix_tokens
        t1 = int(wl.context_lens[s])
        if t1 <= t0:
            continue
        # a tail that starts inside a partial prefix block lands in the
        # sequence's own copy of that block (its table entry after the fork)
        slots = slots_for(tb.tables[s], t0, t1, bs)
        _scatter(_bits(wl.seq_kv("k", s, t0, t1)), _bits(wl.seq_kv("v", s, t0, t1)), kc, vc, slots,
                 code, ks, vs)
    return kc, vc


def expected_paged(wl, tb=None, caches=None, nthreads=0) -> np.ndarray:
    """fp64 outputs [total_q][Hq][D] of the whole workload via the paged oracle."""
    if tb is None:
        tb = build_tables(wl)
    if caches is None:
        caches = build_cache(wl, tb)
    kc, vc = caches
    code = FP8 if wl.kv_dtype == "fp8" else BF16
    ks, vs = wl.fp8_scales() if code == FP8 else (None, None)
    q = _bits(wl.q_values())
    cu = None if wl.is_decode else wl.cu_q_lens
    return paged_attention(q, kc, vc, tb.tables, wl.context_lens, cu, dtype=code, k_scale=ks,
                           v_scale=vs, scale=wl.scale, nthreads=nthreads)


def _kv_f64(wl, which, s, t1, dequant=None):
    """Logical K or V of sequence s, tokens 0..t1-1, as the cache holds them (fp64).
    For fp8 the bytes are encoded with the workload's scales and decoded with
    ``dequant`` = (k_scales, v_scales) when given (default: the same scales)."""
    x = wl.seq_kv(which, s, 0, t1)
    if wl.kv_dtype != "fp8":
        return x.to(torch.float64).numpy()
    ks, vs = wl.fp8_scales()
    sc = ks if which == "k" else vs
    dec = sc if dequant is None else np.asarray(dequant[0 if which == "k" else 1], np.float32)
    f = x.to(torch.float32).numpy()
    codes = e4m3_encode(f / sc[None, :, None].astype(np.float32))
    return e4m3_decode(codes) * dec[None, :, None].astype(np.float64)


def expected_rows(wl, s: int, rows=None, nthreads=0, dequant=None) -> np.ndarray:
    """fp64 outputs [len(rows)][Hq][D] of query rows ``rows`` (indices within the
    sequence's chunk, default all) of sequence s, from the generator's
    contiguous values -- usable at any workload size.  ``dequant`` replaces the
    scales the fp8 bytes are decoded with (tests use it to model a kernel that
    applies the wrong scales to the right bytes)."""
    n = int(wl.q_lens[s])
    L = int(wl.context_lens[s])
    if rows is None:
        rows = np.arange(n)
    rows = np.asarray(rows, dtype=np.int64)
    cu = wl.cu_q_lens
    out = np.empty((len(rows), wl.num_q_heads, wl.head_dim), dtype=np.float64)
    # group consecutive runs to reuse one contiguous call per run
    i = 0
    while i < len(rows):
        j = i
        while j + 1 < len(rows) and rows[j + 1] == rows[j] + 1:
            j += 1
        r0, r1 = int(rows[i]), int(rows[j]) + 1
        Lsub = L - n + r1                       # keys visible to the last row of the run
        k = _kv_f64(wl, "k", s, Lsub, dequant)
        v = _kv_f64(wl, "v", s, Lsub, dequant)
        q = wl.q_values(np.arange(cu[s] + r0, cu[s] + r1)).to(torch.float64).numpy()
        out[i:j + 1] = contiguous_attention(q, k, v, scale=wl.scale, nthreads=nthreads)
        i = j + 1
    return out
