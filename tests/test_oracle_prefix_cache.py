"""Pins of the prefix-cache model against what the pages state and against
closed-form counts (CPU only)."""
import copy

import numpy as np
import pytest

from oracle.allocator import PoolError, PoolModel
from oracle.prefix_cache import BLOCK, PrefixCacheModel


def _request(cache, tokens, salt=0):
    """A request as a scheduler would run it: reuse the cached prefix, allocate
    blocks for the rest, cache its full blocks, then finish (drop its refs).
    Returns (hit blocks, tokens it had to prefill)."""
    hit = cache.match(tokens, salt)
    need = -(-len(tokens) // BLOCK) - len(hit)
    own = cache.alloc(need)
    blocks = hit + own
    cache.insert(tokens, blocks, salt)
    cache.pool.free(blocks)
    return len(hit), len(tokens) - BLOCK * len(hit)


def _vocab(rng, n):
    return [int(x) for x in rng.integers(3, 128000, size=n)]


def test_block_aligned_reuse_of_a_2000_token_prompt():
    """A 2,000-token shared prompt is 125 full blocks; a second request reuses
    exactly those and prefills only its own tail."""
    rng = np.random.default_rng(1)
    sys_prompt = _vocab(rng, 2000)
    c = PrefixCacheModel(PoolModel(1000))
    h0, pre0 = _request(c, sys_prompt + _vocab(rng, 37))
    assert (h0, pre0) == (0, 2037)
    h1, pre1 = _request(c, sys_prompt + [1] + _vocab(rng, 90))
    assert h1 == 125 and pre1 == 91


def test_partial_block_of_a_shared_prompt_is_not_reused():
    """2,008 shared tokens: block 125 holds 8 shared and 8 differing tokens, so
    matching stops at 125 blocks (matching is block-aligned)."""
    rng = np.random.default_rng(2)
    shared = _vocab(rng, 2008)
    c = PrefixCacheModel(PoolModel(1000))
    _request(c, shared + [1] * 40)
    h, pre = _request(c, shared + [2] * 40)
    assert h == 125 and pre == 2048 - 2000


def test_variable_token_at_the_front_gives_zero_hits_and_the_fix_restores_them():
    rng = np.random.default_rng(3)
    sys_prompt = _vocab(rng, 2000)
    c = PrefixCacheModel(PoolModel(4000))
    hits = [_request(c, [1000 + u] + sys_prompt + _vocab(rng, 50))[0] for u in range(20)]
    assert hits == [0] * 20
    c2 = PrefixCacheModel(PoolModel(4000))
    hits2 = [_request(c2, sys_prompt + [1000 + u] + _vocab(rng, 50))[0] for u in range(20)]
    assert hits2 == [0] + [125] * 19


@pytest.mark.parametrize("n,p,t", [(10, 2000, 300), (7, 500, 17), (32, 1024, 1), (5, 15, 100)])
def test_hit_rate_closed_form(n, p, t):
    """n requests = one p-token shared prefix + a t-token tail whose first token
    is unique: every request after the first hits floor(p/16) blocks."""
    rng = np.random.default_rng(n * p + t)
    shared = _vocab(rng, p)
    c = PrefixCacheModel(PoolModel(n * ((p + t) // BLOCK + 1) + 8))
    for i in range(n):
        _request(c, shared + [200000 + i] + _vocab(rng, t - 1))
    st = c.snapshot()
    assert st["lookups"] == n
    assert st["query_blocks"] == n * ((p + t) // BLOCK)
    assert st["hit_blocks"] == (n - 1) * (p // BLOCK)
    assert st["cached_blocks"] == p // BLOCK + n * ((p + t) // BLOCK - p // BLOCK)


def test_rag_reuse_is_the_system_prompt_only():
    """Retrieved passages differ per query: only the system prompt is reused,
    here 496 of 3,500..9,500 tokens -- between 5 and 15 per cent."""
    rng = np.random.default_rng(4)
    sys_prompt = _vocab(rng, 500)
    c = PrefixCacheModel(PoolModel(20000))
    frac = []
    for q in range(12):
        passages = _vocab(rng, int(rng.integers(3000, 9001)))
        h, _ = _request(c, sys_prompt + passages)
        if q:
            assert h == 31
            frac.append(h * BLOCK / (500 + len(passages)))
    assert 0.05 <= min(frac) and max(frac) <= 0.15


def test_tenant_key_isolates_identical_prompts():
    rng = np.random.default_rng(5)
    prompt = _vocab(rng, 640)
    c = PrefixCacheModel(PoolModel(200))
    _request(c, prompt, salt=11)
    assert _request(c, prompt, salt=12)[0] == 0          # another tenant: no match
    assert _request(c, prompt, salt=11)[0] == 40         # same tenant: all 40 blocks


def test_refcounts_cache_holds_one_reference_per_block():
    rng = np.random.default_rng(6)
    prompt = _vocab(rng, 100)                          # 6 full blocks + 4 tokens
    pool = PoolModel(50)
    c = PrefixCacheModel(pool)
    blocks = c.alloc(7)
    assert c.insert(prompt, blocks) == 6                # the partial block is not cached
    assert [pool.ref[b] for b in blocks] == [2] * 6 + [1]
    pool.free(blocks)                                   # the request finishes
    assert [pool.ref[b] for b in blocks] == [1] * 6 + [0]
    a = c.match(prompt)
    b = c.match(prompt[:64])
    assert a == blocks[:6] and b == blocks[:4]
    assert [pool.ref[x] for x in blocks[:6]] == [3, 3, 3, 3, 2, 2]


def test_duplicate_insert_keeps_the_first_copy():
    rng = np.random.default_rng(7)
    prompt = _vocab(rng, 64)
    pool = PoolModel(50)
    c = PrefixCacheModel(pool)
    a, b = c.alloc(4), c.alloc(4)                       # two requests computed it concurrently
    assert c.insert(prompt, a) == 4
    assert c.insert(prompt, b) == 0
    assert [pool.ref[x] for x in a] == [2] * 4 and [pool.ref[x] for x in b] == [1] * 4
    assert c.match(prompt) == a


def _tree():
    """Trunk S (4 blocks) with branches A and B (2 blocks each)."""
    rng = np.random.default_rng(8)
    S, A, B = _vocab(rng, 64), _vocab(rng, 32), _vocab(rng, 32)
    pool = PoolModel(64)
    c = PrefixCacheModel(pool)
    sa = c.alloc(6)
    c.insert(S + A, sa)                                 # clock 1
    pool.free(sa)
    hb = c.match(S + B)                                 # clock 2: the trunk
    ob = c.alloc(2)
    c.insert(S + B, hb + ob)                            # clock 3
    pool.free(hb + ob)
    return c, S, A, B, sa, ob


def test_eviction_is_lru_over_leaves():
    c, S, A, B, sa, ob = _tree()
    c.pool.free(c.match(S + A))                         # clock 4: A is now the most recent
    freed = c.evict(100)
    # B's blocks (clock 3) leave before A's (clock 4), each branch from its end;
    # the trunk (clock 4, inserted before A) goes last, from its end
    assert freed == [ob[1], ob[0], sa[5], sa[4], sa[3], sa[2], sa[1], sa[0]]
    assert c.cached_blocks == 0 and c.pool.free_blocks == 64


def test_eviction_skips_blocks_a_request_still_holds():
    c, S, A, B, sa, ob = _tree()
    held = c.match(S + A)                               # a live request on S + A
    assert c.evictable_blocks() == 2
    freed = c.evict(100)
    assert freed == [ob[1], ob[0]]                      # the trunk is in use, and so is A
    c.pool.free(held)                                   # the request ends
    assert c.evictable_blocks() == 6
    assert len(c.evict(100)) == 6


def test_trunk_outlives_its_branches():
    """One system prompt at the root, per-step branches off it: evicting as many
    blocks as the branches hold frees the branches only."""
    rng = np.random.default_rng(9)
    trunk = _vocab(rng, 320)                            # 20 blocks
    c = PrefixCacheModel(PoolModel(400))
    for _ in range(10):
        _request(c, trunk + _vocab(rng, 48))            # 3 branch blocks each
    assert c.cached_blocks == 20 + 30
    c.evict(30)
    assert c.cached_blocks == 20
    assert _request(c, trunk + [5] * 16)[0] == 20


def test_alloc_evicts_only_the_shortfall():
    rng = np.random.default_rng(10)
    pool = PoolModel(20)
    c = PrefixCacheModel(pool)
    prompt = _vocab(rng, 160)
    blocks = c.alloc(10)
    c.insert(prompt, blocks)
    pool.free(blocks)
    assert pool.free_blocks == 10 and c.cached_blocks == 10
    got = c.alloc(15)
    assert c.stats["evicted_blocks"] == 5 and c.cached_blocks == 5
    assert got[:5] == blocks[5:]                        # evicted 9, 8, .., 5; LIFO hands 5 out first
    assert c.match(prompt) == blocks[:5]


def test_alloc_failure_after_eviction():
    rng = np.random.default_rng(11)
    pool = PoolModel(8)
    c = PrefixCacheModel(pool)
    blocks = c.alloc(8)
    c.insert(_vocab(rng, 128), blocks)
    pool.free(blocks[4:])
    held = blocks[:4]                                   # a live request keeps the first 4
    with pytest.raises(PoolError) as e:
        c.alloc(8)
    assert e.value.status == 2
    assert c.cached_blocks == 4 and pool.free_blocks == 4
    pool.free(held)


def test_evictable_count_agrees_with_exhaustive_eviction():
    rng = np.random.default_rng(12)
    pool = PoolModel(300)
    c = PrefixCacheModel(pool)
    trunks = [_vocab(rng, 48) for _ in range(3)]
    live = []
    for i in range(25):
        toks = trunks[i % 3] + _vocab(rng, int(rng.integers(0, 70)))
        hit = c.match(toks)
        own = c.alloc(-(-len(toks) // BLOCK) - len(hit))
        c.insert(toks, hit + own)
        if i % 4 == 0:
            live.append(hit + own)                      # still running
        else:
            pool.free(hit + own)
    c2 = copy.deepcopy(c)
    assert c.evictable_blocks() == len(c2.evict(10 ** 6))
