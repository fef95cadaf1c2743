"""Swap-out / swap-in of KV blocks to host memory, as plain array operations
(test infrastructure only; nothing in the library imports it).

When the cache runs out mid-generation the scheduler may preempt a request
and ship its blocks to host memory, bringing them back later ("Waste, and
three ways to reclaim it", "When it runs out anyway": swap to host memory;
"M.65 Inference serving", block management (f) preemption: swap out to CPU).
The blocks come back wherever the pool has room, so the block table is
rewritten; the bytes of every (block, KV head) tile must survive unchanged.

* swap-out of ids[0..n): host[i] = cache[ids[i]] for both caches, i.e. the
  host buffer is [n][Hkv][16][128] in list order;
* swap-in into new ids: cache[new_ids[i]] = host[i] (ids distinct).
"""
from __future__ import annotations

import numpy as np


def swap_out(k_cache: np.ndarray, v_cache: np.ndarray, ids) -> tuple[np.ndarray, np.ndarray]:
    ids = np.asarray(ids, dtype=np.int64)
    if ids.size and (ids.min() < 0 or ids.max() >= k_cache.shape[0]):
        raise IndexError("block id outside the pool")
    return k_cache[ids].copy(), v_cache[ids].copy()


def swap_in(k_cache: np.ndarray, v_cache: np.ndarray, ids, host_k: np.ndarray, host_v: np.ndarray) -> None:
    ids = np.asarray(ids, dtype=np.int64)
    if len(set(ids.tolist())) != ids.size:
        raise ValueError("swap-in ids must be distinct")
    if ids.size and (ids.min() < 0 or ids.max() >= k_cache.shape[0]):
        raise IndexError("block id outside the pool")
    k_cache[ids] = host_k
    v_cache[ids] = host_v
