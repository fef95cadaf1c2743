"""Python model of the block-hash prefix cache and its LRU eviction
(test infrastructure only; nothing in the library imports it).

What it models, restated from the pages:

* Prefix caching keeps the KV blocks of a prompt prefix after the request that
  computed them has finished, so a later request starting with the same tokens
  reuses them instead of prefilling again.  ["PagedAttention, chunked prefill,
  and the launch that cascades", opening section: hash the prefix and reuse the
  computed blocks across requests; "Waste, and three ways to reclaim it",
  "Block sharing versus prefix caching?": sharing is between live requests,
  prefix caching keeps blocks after a request ends.]
* Matching is on exact token ids, block-aligned, from the very start: a
  difference anywhere invalidates every block after it, so a variable token at
  the front gives zero hits.  ["Waste, and three ways to reclaim it", "Why does
  my prefix cache hit rate not match what I expect?"; "PagedAttention, chunked
  prefill, ...", prefix cache thrashing.]
* The cache is keyed per tenant, so one tenant's blocks cannot be matched by
  another's request.  ["Waste, and three ways to reclaim it", "The isolation
  question".]
* Finished requests' blocks are kept in a tree organised by shared beginnings
  and evicted least recently used first; a new request walks down from the
  root as far as it matches and prefills only the rest.  ["Waste, and three
  ways to reclaim it", "SGLang -- RadixAttention" and the LRU radix tree of
  "vLLM or SGLang, and why?".]

The definition used here is the plainest one: the cached block j of a token
sequence under tenant key ``salt`` is keyed by ``(salt, tokens[0 : 16 (j+1)])``
-- every token from the start through the end of that block.  Only full blocks
are cached.  The cache holds one pool reference per cached block.

Readings where the pages are silent (the library takes the same ones):

* Recency: every call (match or insert) advances a clock by one; every cached
  block the call matches or inserts takes the clock's value.
* Eviction takes, one block at a time, the cached block with the oldest
  recency (ties: the one cached first) among those that (a) no longer entry
  extends (a leaf of the tree: evicting an inner block would strand the blocks
  after it, which can only be matched through it) and (b) only the cache holds
  (pool refcount 1: "evict at refcount 0" once the cache's own reference is
  discounted).
* Insert keeps an existing entry for the same key (it does not swap in the
  caller's physical block); it caches at most ``min(len(tokens) // 16,
  len(block_ids))`` blocks.
* ``alloc`` evicts exactly the shortfall (as far as possible) before
  allocating from the pool; if the pool is still short it fails, and the
  evictions it made stand.
"""
from __future__ import annotations

from dataclasses import dataclass

from oracle.allocator import ERR_INVALID, ERR_OUT_OF_BLOCKS, PoolError, PoolModel

BLOCK = 16


@dataclass
class _Entry:
    block: int
    tick: int
    serial: int


class PrefixCacheModel:
    def __init__(self, pool: PoolModel):
        self.pool = pool
        self.entries: dict[tuple, _Entry] = {}
        self.clock = 0
        self.serial = 0
        self.stats = {"lookups": 0, "query_blocks": 0, "hit_blocks": 0, "inserted_blocks": 0,
                      "evicted_blocks": 0}

    # --------------------------------------------------------------- helpers
    @staticmethod
    def _key(salt: int, tokens, j: int) -> tuple:
        return (int(salt), tuple(int(t) for t in tokens[: BLOCK * (j + 1)]))

    def _is_leaf(self, key: tuple) -> bool:
        salt, toks = key
        n = len(toks)
        for s2, t2 in self.entries:
            if s2 == salt and len(t2) == n + BLOCK and t2[:n] == toks:
                return False
        return True

    # ------------------------------------------------------------------- ops
    def match(self, tokens, salt: int = 0) -> list[int]:
        """Longest run of cached full blocks from the start; the caller gets one
        reference to each returned block."""
        self.clock += 1
        nfull = len(tokens) // BLOCK
        out = []
        for j in range(nfull):
            e = self.entries.get(self._key(salt, tokens, j))
            if e is None:
                break
            e.tick = self.clock
            out.append(e.block)
        self.pool.share(out)
        self.stats["lookups"] += 1
        self.stats["query_blocks"] += nfull
        self.stats["hit_blocks"] += len(out)
        return out

    def insert(self, tokens, block_ids, salt: int = 0) -> int:
        """Caches the full blocks of ``tokens`` held in ``block_ids`` (the
        caller's blocks, in logical order); returns how many were new."""
        n = min(len(tokens) // BLOCK, len(block_ids))
        for b in block_ids[:n]:
            if b < 0 or b >= self.pool.num_blocks or self.pool.ref[b] < 1:
                raise PoolError(ERR_INVALID, "insert of a block that is not live")
        self.clock += 1
        new = 0
        for j in range(n):
            key = self._key(salt, tokens, j)
            e = self.entries.get(key)
            if e is not None:
                e.tick = self.clock
                continue
            self.pool.share([int(block_ids[j])])
            self.entries[key] = _Entry(int(block_ids[j]), self.clock, self.serial)
            self.serial += 1
            new += 1
        self.stats["inserted_blocks"] += new
        return new

    def evict(self, n: int) -> list[int]:
        """Frees up to n cached blocks, least recently used evictable leaf first."""
        if n < 0:
            raise PoolError(ERR_INVALID, "n < 0")
        freed = []
        while len(freed) < n:
            cands = [k for k, e in self.entries.items()
                     if self.pool.ref[e.block] == 1 and self._is_leaf(k)]
            if not cands:
                break
            k = min(cands, key=lambda k: (self.entries[k].tick, self.entries[k].serial))
            b = self.entries.pop(k).block
            self.pool.free([b])
            freed.append(b)
        self.stats["evicted_blocks"] += len(freed)
        return freed

    def alloc(self, n: int) -> list[int]:
        if n < 0:
            raise PoolError(ERR_INVALID, "n < 0")
        short = n - self.pool.free_blocks
        if short > 0:
            self.evict(short)
        return self.pool.alloc(n)

    # ----------------------------------------------------------------- views
    @property
    def cached_blocks(self) -> int:
        return len(self.entries)

    def evictable_blocks(self) -> int:
        """Blocks that repeated eviction could free now (only the cache holds them
        and every entry below them is evictable too)."""
        # an entry is evictable-eventually iff its block has refcount 1 and all of
        # its descendants are evictable-eventually
        keys = sorted(self.entries, key=lambda k: -len(k[1]))   # deepest first
        ok: dict[tuple, bool] = {}
        for k in keys:
            salt, toks = k
            kids_ok = all(ok[k2] for k2 in ok if k2[0] == salt and len(k2[1]) == len(toks) + BLOCK
                          and k2[1][: len(toks)] == toks)
            ok[k] = kids_ok and self.pool.ref[self.entries[k].block] == 1
        return sum(ok.values())

    def snapshot(self) -> dict:
        return dict(self.stats, cached_blocks=self.cached_blocks)


__all__ = ["PrefixCacheModel", "BLOCK", "ERR_INVALID", "ERR_OUT_OF_BLOCKS", "PoolError"]
