"""Puts a synthetic workload on the device through the library's own calls.

This is the scheduler-side driver a server would run around the library:
block tables come from the library's block manager (kv_pool), the cache is
filled with reshape_and_cache, copy-on-write forks use kv_copy_on_write's
device copy, and one layer step is ``reshape_and_cache`` of the step's new
tokens followed by paged attention (decode, or the mixed chunked-prefill call).
Slot numbers are the scheduler's bookkeeping: token t of a sequence lives in
block table[t // 16] at offset t % 16.
"""
from __future__ import annotations

import numpy as np
import torch

from . import (KVPool, paged_attention_chunked_prefill, paged_attention_chunked_prefill_workspace_size,
               paged_attention_decode, paged_attention_workspace_size, reshape_and_cache)

FILL_CHUNK_TOKENS = 1 << 15


def _blocks(n, bs=16):
    return -(-int(n) // bs)


class DeviceWorkload:
    """A workload resident in HBM, ready to run layer steps."""

    def __init__(self, wl, device="cuda", poison_cache=False):
        self.wl = wl
        self.device = torch.device(device)
        B, mb, bs = wl.num_seqs, wl.max_blocks_per_seq, wl.block_size
        self.pool = KVPool(wl.num_blocks, wl.free_order)
        cache_dtype = torch.uint8 if wl.kv_dtype == "fp8" else torch.bfloat16
        shape = (wl.num_blocks, wl.num_kv_heads, bs, wl.head_dim)
        if poison_cache:
            # every byte 0xFF: NaN in bf16 and in e4m3, so any read of a slot that
            # was never written shows up in the output
            if cache_dtype == torch.bfloat16:
                self.k_cache = torch.full(shape, -1, dtype=torch.int16, device=self.device).view(cache_dtype)
            else:
                self.k_cache = torch.full(shape, 255, dtype=torch.uint8, device=self.device)
            self.v_cache = self.k_cache.clone()
        else:
            self.k_cache = torch.zeros(shape, dtype=cache_dtype, device=self.device)
            self.v_cache = torch.zeros(shape, dtype=cache_dtype, device=self.device)
        if wl.kv_dtype == "fp8":
            ks, vs = wl.fp8_scales(device=self.device)
            self.k_scale = torch.from_numpy(ks).to(self.device)
            self.v_scale = torch.from_numpy(vs).to(self.device)
        else:
            self.k_scale = self.v_scale = None
        tables = np.full((B, mb), -1, dtype=np.int32)
        pb = _blocks(wl.prefix_tokens, bs) if wl.prefix_tokens else 0
        if pb:
            pre = self.pool.alloc(pb)
            tables[0, :pb] = pre
            for s in range(1, B):
                self.pool.share(pre)
                tables[s, :pb] = pre
            row = np.full(mb, -1, dtype=np.int32)
            row[:pb] = pre
            self._write_tokens([(0, 0, wl.prefix_tokens)], {0: row})
        if wl.cow_block >= 0:
            for s in range(B):
                tables[s, wl.cow_block] = self.pool.copy_on_write(int(tables[s, wl.cow_block]),
                                                                  self.k_cache, self.v_cache)
        for s in range(B):
            n = _blocks(int(wl.context_lens[s]), bs) - pb
            tables[s, pb:pb + n] = self.pool.alloc(n)
        self.tables_host = tables
        # history: every token before the step's new ones
        hist = []
        for s in range(B):
            t0 = wl.prefix_tokens
            t1 = int(wl.context_lens[s]) - int(wl.q_lens[s])
            if t1 > t0:
                hist.append((s, t0, t1))
        self._write_tokens(hist, {s: tables[s] for s in range(B)})
        # step inputs
        new = [(s, int(wl.context_lens[s]) - int(wl.q_lens[s]), int(wl.context_lens[s])) for s in range(B)]
        keys = np.concatenate([wl.token_keys(s, a, b) for s, a, b in new])
        slots = np.concatenate([self._slots(tables[s], a, b) for s, a, b in new])
        self.new_k = wl.kv_values("k", keys, self.device)
        self.new_v = wl.kv_values("v", keys, self.device)
        self.slot_mapping = torch.from_numpy(slots).to(self.device)
        self.q = wl.q_values(device=self.device)
        self.block_tables = torch.from_numpy(tables).to(self.device)
        self.context_lens = torch.from_numpy(wl.context_lens).to(self.device)
        self.cu_q_lens = torch.from_numpy(wl.cu_q_lens).to(self.device)
        self.out = torch.empty(wl.total_q, wl.num_q_heads, wl.head_dim, dtype=torch.float32, device=self.device)
        if wl.is_decode:
            nbytes = paged_attention_workspace_size(B, wl.num_q_heads, mb, wl.num_splits)
        else:
            nbytes = paged_attention_chunked_prefill_workspace_size(
                B, wl.total_q, int(wl.q_lens.max()), wl.num_q_heads, wl.num_kv_heads, mb, wl.num_splits)
        self.workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=self.device) if nbytes else None
        torch.cuda.synchronize(self.device)

    @staticmethod
    def _slots(row, t0, t1, bs=16):
        t = np.arange(t0, t1, dtype=np.int64)
        return row[t // bs].astype(np.int64) * bs + t % bs

    def _write_tokens(self, spans, rows):
        """reshape_and_cache of the given (seq, t0, t1) spans, in chunks."""
        wl = self.wl
        buf_keys, buf_slots, n = [], [], 0

        def flush():
            nonlocal buf_keys, buf_slots, n
            if not n:
                return
            keys = np.concatenate(buf_keys)
            slots = torch.from_numpy(np.concatenate(buf_slots)).to(self.device)
            k = wl.kv_values("k", keys, self.device)
            v = wl.kv_values("v", keys, self.device)
            reshape_and_cache(k, v, self.k_cache, self.v_cache, slots, self.k_scale, self.v_scale)
            buf_keys, buf_slots, n = [], [], 0

        for s, t0, t1 in spans:
            a = t0
            while a < t1:
                b = min(t1, a + FILL_CHUNK_TOKENS - n)
                buf_keys.append(wl.token_keys(s, a, b))
                buf_slots.append(self._slots(rows[s], a, b))
                n += b - a
                a = b
                if n >= FILL_CHUNK_TOKENS:
                    flush()
        flush()

    # ------------------------------------------------------------- one step
    def write_new_tokens(self, stream=None):
        reshape_and_cache(self.new_k, self.new_v, self.k_cache, self.v_cache, self.slot_mapping,
                          self.k_scale, self.v_scale, stream=stream)

    def attention(self, stream=None):
        wl = self.wl
        if wl.is_decode:
            return paged_attention_decode(self.out, self.q, self.k_cache, self.v_cache, self.block_tables,
                                          self.context_lens, wl.scale, self.k_scale, self.v_scale,
                                          wl.num_splits, self.workspace, stream=stream)
        return paged_attention_chunked_prefill(self.out, self.q, self.cu_q_lens, self.context_lens,
                                               int(wl.q_lens.max()), self.k_cache, self.v_cache,
                                               self.block_tables, wl.scale, self.k_scale, self.v_scale,
                                               wl.num_splits, self.workspace, stream=stream)

    def step(self, stream=None):
        self.write_new_tokens(stream)
        return self.attention(stream)
