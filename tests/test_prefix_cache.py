"""The library's prefix cache (C++, through the C ABI) against the Python model
of the same rules, operation by operation: block ids, eviction order, pool
refcounts and statistics must agree exactly (CPU only, no GPU needed)."""
import numpy as np
import pytest

import paged_kv_cache_263_gb300 as pkv
from oracle.allocator import PoolError, PoolModel
from oracle.prefix_cache import BLOCK, PrefixCacheModel


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_cache_263_gb300 import build
    build.build()


def _pair(num_blocks, order=None):
    pool = pkv.KVPool(num_blocks, order)
    return pool, pkv.PrefixCache(pool), PrefixCacheModel(PoolModel(num_blocks, order))


def _same_pool(pool, model, num_blocks):
    assert [pool.refcount(b) for b in range(num_blocks)] == model.pool.ref
    st = pool.stats()
    assert st["free"] == model.pool.free_blocks


def _same_stats(cache, model):
    st = cache.stats()
    ms = model.snapshot()
    for k in ("lookups", "query_blocks", "hit_blocks", "inserted_blocks", "evicted_blocks", "cached_blocks"):
        assert st[k] == ms[k], k
    assert st["evictable_blocks"] == model.evictable_blocks()


@pytest.mark.parametrize("seed,nb", [(0, 160), (1, 160), (2, 48), (3, 40)])
def test_random_traffic_matches_the_model(seed, nb):
    """Agent-loop / multi-turn traffic over a few tenants and system prompts:
    every call's result, the pool's refcounts and the statistics agree.  The
    small pools run out of blocks, so allocation failures are covered too."""
    rng = np.random.default_rng(100 + seed)
    order = rng.permutation(nb).astype(np.int32)
    pool, cache, model = _pair(nb, order)
    trunks = [[int(x) for x in rng.integers(0, 50000, size=int(rng.integers(16, 120)))] for _ in range(4)]
    live = []                                               # requests still holding blocks
    for step in range(400):
        op = rng.random()
        if op < 0.55:
            t = trunks[int(rng.integers(0, 4))]
            salt = int(rng.integers(0, 2))
            cut = int(rng.integers(0, len(t) + 1))
            toks = t[:cut] + [int(x) for x in rng.integers(0, 50000, size=int(rng.integers(0, 60)))]
            cap = None if rng.random() < 0.8 else int(rng.integers(0, 8))
            got = cache.match(toks, salt, cap).tolist()
            want = model.match(toks if cap is None else toks[: BLOCK * cap], salt)
            assert got == want
            need = -(-len(toks) // BLOCK) - len(got)
            try:
                own = model.alloc(need)
            except PoolError:
                with pytest.raises(pkv.KVError):
                    cache.alloc(need)
                pool.free(got)
                model.pool.free(want)
                continue
            assert cache.alloc(need).tolist() == own
            blocks = got + own
            assert cache.insert(toks, blocks, salt) == model.insert(toks, blocks, salt)
            if rng.random() < 0.3:
                live.append(blocks)
            else:
                pool.free(blocks)
                model.pool.free(blocks)
        elif op < 0.75 and live:
            blocks = live.pop(int(rng.integers(0, len(live))))
            pool.free(blocks)
            model.pool.free(blocks)
        else:
            n = int(rng.integers(0, 12))
            assert cache.evict(n).tolist() == model.evict(n)
        if step % 25 == 0:
            _same_pool(pool, model, nb)
            _same_stats(cache, model)
    _same_pool(pool, model, nb)
    _same_stats(cache, model)
    for blocks in live:
        pool.free(blocks)
        model.pool.free(blocks)
    assert cache.evict(10 ** 6).tolist() == model.evict(10 ** 6)
    assert cache.stats()["cached_blocks"] == 0 and pool.stats()["free"] == nb


def test_thrash_case_through_the_library():
    rng = np.random.default_rng(7)
    sys_prompt = [int(x) for x in rng.integers(0, 50000, size=2000)]
    pool, cache, _ = _pair(4000)
    hits = []
    for u in range(10):
        toks = [90000 + u] + sys_prompt + [1, 2, 3]
        h = cache.match(toks)
        own = cache.alloc(-(-len(toks) // BLOCK) - len(h))
        cache.insert(toks, np.concatenate([h, own]))
        pool.free(np.concatenate([h, own]))
        hits.append(len(h))
    assert hits == [0] * 10
    st = cache.stats()
    assert st["hit_blocks"] == 0 and st["cached_blocks"] == 10 * 125


def test_tenant_keys_and_64_bit_salts():
    rng = np.random.default_rng(8)
    toks = [int(x) for x in rng.integers(0, 50000, size=64)]
    pool, cache, _ = _pair(64)
    b = cache.alloc(4)
    cache.insert(toks, b, salt=2**64 - 1)
    pool.free(b)
    assert cache.match(toks, salt=2**63 - 1).size == 0
    got = cache.match(toks, salt=2**64 - 1)
    assert got.tolist() == b.tolist()
    pool.free(got)


def test_insert_rejects_free_blocks_and_changes_nothing():
    pool, cache, _ = _pair(8)
    b = cache.alloc(2)
    with pytest.raises(pkv.KVError) as e:
        cache.insert(list(range(48)), [int(b[0]), int(b[1]), 5])   # block 5 is free
    assert e.value.status == 1
    st = cache.stats()
    assert st["cached_blocks"] == 0 and st["inserted_blocks"] == 0
    assert [pool.refcount(x) for x in b] == [1, 1]


def test_destroy_releases_the_cache_references():
    pool, cache, _ = _pair(16)
    b = cache.alloc(3)
    cache.insert(list(range(48)), b)
    pool.free(b)
    assert pool.stats()["free"] == 13
    cache.close()
    assert pool.stats()["free"] == 16


def test_waste_stats_match_the_model():
    from oracle.allocator import waste_stats
    rng = np.random.default_rng(21)
    for n, res in ((4, 8192), (100, 32768), (1, 16), (0, 100)):
        lens = rng.integers(0, res + 1, size=n)
        got = pkv.kv_waste_stats(lens, res)
        want = waste_stats(lens, res)
        for k, v in want.items():
            assert got[k] == pytest.approx(v, rel=1e-12, abs=1e-12), k
    got = pkv.kv_waste_stats([300, 2000, 600, 4400], 8192)
    assert got["contiguous_untouched_slots"] == 25468 and got["paged_waste_slots"] == 12
    with pytest.raises(pkv.KVError):
        pkv.kv_waste_stats([9000], 8192)
