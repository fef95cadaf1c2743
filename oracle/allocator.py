"""Python model of the paged block manager (test infrastructure only).

Rules, restated from the pages:

* The pool is a set of fixed-size physical blocks; allocation takes blocks
  from a free list in O(1) and a finished request returns all its blocks.
  ["M.65 Inference serving", PagedAttention block management (c)];
  ["PagedAttention, chunked prefill, and the launch that cascades",
  section "PagedAttention: an OS idea, not an ML one"].
* Shared prefix blocks are reference-counted: two sharers -> refcount 2, a
  release decrements, at 0 the block returns to the pool.
  ["M.65 Inference serving", block management (e)]; ["Waste, and three ways
  to reclaim it", section "Sharing, and what makes a prefix reusable"].
* Copy-on-write: a sequence about to write into a shared block first gets its
  own copy.  ["Waste, and three ways to reclaim it", "Copy on write"];
  ["M.65 Inference serving", block management (g)].

The pages do not fix the free-list order.  The reading used here (and by the
library) is a LIFO stack: ``initial_free_order[0]`` is handed out first, a freed
block is the next one handed out.  Allocation is all-or-nothing.
"""
from __future__ import annotations

from collections import Counter

OK, ERR_INVALID, ERR_OUT_OF_BLOCKS = 0, 1, 2


class PoolError(Exception):
    def __init__(self, status, msg=""):
        super().__init__(msg or {1: "invalid", 2: "out of blocks"}.get(status, str(status)))
        self.status = status


class PoolModel:
    def __init__(self, num_blocks: int, initial_free_order=None):
        if num_blocks < 1:
            raise PoolError(ERR_INVALID, "num_blocks")
        order = list(range(num_blocks)) if initial_free_order is None else [int(x) for x in initial_free_order]
        if sorted(order) != list(range(num_blocks)):
            raise PoolError(ERR_INVALID, "initial_free_order must be a permutation")
        self.num_blocks = num_blocks
        self._stack = order[::-1]           # top of stack = next block handed out
        self.ref = [0] * num_blocks
        self.cow_copies = 0
        self.alloc_failures = 0

    # ------------------------------------------------------------------ ops
    def alloc(self, n: int) -> list[int]:
        if n < 0:
            raise PoolError(ERR_INVALID, "n < 0")
        if n > len(self._stack):
            self.alloc_failures += 1
            raise PoolError(ERR_OUT_OF_BLOCKS)
        ids = [self._stack.pop() for _ in range(n)]
        for b in ids:
            self.ref[b] = 1
        return ids

    def _check_live(self, ids, need=None):
        cnt = Counter(int(b) for b in ids)
        for b, c in cnt.items():
            if b < 0 or b >= self.num_blocks or self.ref[b] < (c if need is None else need):
                raise PoolError(ERR_INVALID, f"block {b} not live enough")

    def free(self, ids) -> None:
        self._check_live(ids)
        for b in ids:
            b = int(b)
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self._stack.append(b)

    def share(self, ids) -> None:
        self._check_live(ids, need=1)
        for b in ids:
            self.ref[int(b)] += 1

    def copy_on_write(self, b: int) -> tuple[int, bool]:
        """Returns (block to write into, whether its contents must be copied)."""
        b = int(b)
        if b < 0 or b >= self.num_blocks or self.ref[b] < 1:
            raise PoolError(ERR_INVALID, "cow of a free block")
        if self.ref[b] == 1:
            return b, False
        (nb,) = self.alloc(1)
        self.ref[b] -= 1
        self.cow_copies += 1
        return nb, True

    # ---------------------------------------------------------------- stats
    @property
    def free_blocks(self) -> int:
        return len(self._stack)

    def stats(self) -> dict:
        live = sum(1 for r in self.ref if r > 0)
        shared = sum(1 for r in self.ref if r > 1)
        return {"free": len(self._stack), "live": live, "shared": shared,
                "cow_copies": self.cow_copies, "alloc_failures": self.alloc_failures}

    def free_list(self) -> list[int]:
        """Blocks in the order they would be handed out next."""
        return self._stack[::-1]


def blocks_for(tokens: int, block_size: int = 16) -> int:
    """Number of blocks a sequence of ``tokens`` tokens occupies (ceil division)."""
    return -(-int(tokens) // block_size)


def waste_stats(lens, reservation_tokens: int, block_size: int = 16) -> dict:
    """Memory waste of a set of requests, contiguous against paged
    ["Waste, and three ways to reclaim it", "PagedAttention" (the worked example:
    four requests each reserving a whole maximum-length buffer) and "Small block
    size" (internal waste capped at block_size - 1 tokens per sequence)].

    Contiguous: every request reserves ``reservation_tokens`` slots; the slots no
    token uses are untouched.  Paged: every request holds ceil(len / block_size)
    blocks; the unused slots of its last block are the internal waste."""
    lens = [int(x) for x in lens]
    if any(L < 0 or L > reservation_tokens for L in lens) or reservation_tokens < 0:
        raise PoolError(ERR_INVALID, "length outside the reservation")
    used = sum(lens)
    reserved = reservation_tokens * len(lens)
    blocks = sum(blocks_for(L, block_size) for L in lens)
    slots = blocks * block_size
    return {
        "used_tokens": used,
        "contiguous_reserved_slots": reserved,
        "contiguous_untouched_slots": reserved - used,
        "contiguous_untouched_percent": 100.0 * (reserved - used) / reserved if reserved else 0.0,
        "paged_blocks": blocks,
        "paged_slots": slots,
        "paged_waste_slots": slots - used,
        "paged_waste_percent": 100.0 * (slots - used) / slots if slots else 0.0,
    }
