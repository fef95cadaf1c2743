"""Pins for the block-manager model and the sizing arithmetic the pages print."""
import numpy as np
import pytest

from oracle.allocator import ERR_INVALID, ERR_OUT_OF_BLOCKS, PoolError, PoolModel, blocks_for, waste_stats


def test_worked_allocation_example(golden):
    kv, _ = golden("worked_allocation_example.txt")
    used = [int(x) for x in kv["used_tokens"].split()]
    limit = int(kv["reservation_tokens"])
    bs = int(kv["block_size"])
    lo, hi = (int(x) for x in kv["waste_band_percent"].split())
    reserved = limit * len(used)
    untouched = reserved - sum(used)
    assert (reserved, untouched) == (32768, 25468)
    pct = 100.0 * untouched / reserved
    assert abs(pct - 77.72) < 0.01
    assert lo <= pct <= hi                      # inside the pages' 60-80% band
    # the printed 63% does not follow from the printed counts
    assert abs(pct - int(kv["printed_untouched_percent"])) > 10
    # contiguous: a fifth 8,192 reservation does not fit in a 32,768-slot pool
    assert reserved + limit > 4 * limit
    # paged: the same four requests take 457 blocks, 12 slots of internal waste
    nblk = [blocks_for(u, bs) for u in used]
    assert sum(nblk) == 457 and sum(nblk) * bs - sum(used) == 12
    pool = PoolModel(reserved // bs)
    for n in nblk:
        pool.alloc(n)
    pool.alloc(blocks_for(limit, bs))           # the fifth request is admitted
    assert pool.free_blocks == 2048 - 457 - 512


def test_internal_waste_is_at_most_15_tokens(golden):
    kv, _ = golden("block_table_figures.txt")
    bs = int(kv["block_size"])
    cap = int(kv["max_internal_waste_tokens"])
    rng = np.random.default_rng(0)
    lens = rng.integers(1, 200_000, size=100_000)
    waste = np.array([blocks_for(L, bs) * bs - L for L in lens])
    assert waste.max() <= cap == bs - 1
    assert (waste == cap).any()


def test_block_table_length_for_500_tokens(golden):
    kv, _ = golden("block_table_figures.txt")
    assert blocks_for(500, int(kv["block_size"])) == int(kv["tokens_500_block_ids"])
    assert blocks_for(512) == 32 and blocks_for(513) == 33 and blocks_for(1) == 1


def test_shared_prompt_saving(golden):
    kv, _ = golden("block_table_figures.txt")
    layers, hkv, d, nbytes = (int(x) for x in kv["llama3_8b_shape"].split())
    per_token = 2 * layers * hkv * d * nbytes
    assert per_token == 131072
    saving = int(kv["shared_prompt_tokens"]) * per_token / 2 ** 30
    assert round(saving, 2) == float(kv["saving_per_request_gib"])
    total = saving * int(kv["requests"])
    assert abs(total - int(kv["total_without_sharing_gib"])) / 120 < 0.03   # 122.07 GiB


def test_kv_size_formula(golden):
    _, rows = golden("kv_size_formula.txt")
    seen = {}
    for name, layers, heads, d, seq, nbytes, printed, unit in rows:
        b = 2 * int(layers) * int(heads) * int(d) * int(seq) * int(nbytes)
        val = b / {"MB": 1e6, "GB": 1e9}[unit]
        seen[name] = b
        assert abs(val - float(printed)) / float(printed) < 0.08, (name, val)
    assert seen["llama70b_mha_per_token"] == 2621440
    # 128K with GQA: 42.9e9 bytes = 40 GiB, the page's "roughly 41GB"
    assert seen["llama3_70b_gqa_128k"] == 42949672960 == 40 * 2 ** 30


def test_lifo_order_and_initial_order():
    pool = PoolModel(6, [3, 5, 0, 1, 4, 2])
    assert pool.alloc(2) == [3, 5]
    assert pool.alloc(1) == [0]
    pool.free([5])
    assert pool.alloc(2) == [5, 1]
    assert pool.free_list() == [4, 2]


def test_alloc_is_all_or_nothing():
    pool = PoolModel(4)
    pool.alloc(3)
    before = (pool.free_list(), list(pool.ref))
    with pytest.raises(PoolError) as e:
        pool.alloc(2)
    assert e.value.status == ERR_OUT_OF_BLOCKS
    assert (pool.free_list(), list(pool.ref)) == before
    assert pool.stats()["alloc_failures"] == 1


def test_refcount_lifecycle():
    pool = PoolModel(8)
    (b,) = pool.alloc(1)
    pool.share([b])
    assert pool.ref[b] == 2 and pool.stats()["shared"] == 1
    pool.free([b])
    assert pool.ref[b] == 1 and b not in pool.free_list()
    pool.free([b])
    assert pool.ref[b] == 0 and pool.free_list()[0] == b
    with pytest.raises(PoolError) as e:
        pool.free([b])
    assert e.value.status == ERR_INVALID
    with pytest.raises(PoolError):
        pool.share([b])


def test_no_external_fragmentation():
    """Any free block satisfies any request: after arbitrary churn, a request for
    every remaining free block succeeds."""
    rng = np.random.default_rng(3)
    pool = PoolModel(1000, rng.permutation(1000))
    live = []
    for _ in range(2000):
        if live and rng.random() < 0.45:
            seq = live.pop(int(rng.integers(len(live))))
            pool.free(seq)
        else:
            n = int(rng.integers(1, 40))
            if n <= pool.free_blocks:
                live.append(pool.alloc(n))
    rest = pool.alloc(pool.free_blocks)
    assert pool.free_blocks == 0 and len(set(rest)) == len(rest)


def test_copy_on_write_rules():
    pool = PoolModel(8)
    (b,) = pool.alloc(1)
    assert pool.copy_on_write(b) == (b, False)           # sole owner writes in place
    pool.share([b])
    nb, need = pool.copy_on_write(b)
    assert need and nb != b and pool.ref[b] == 1 and pool.ref[nb] == 1
    assert pool.stats()["cow_copies"] == 1
    with pytest.raises(PoolError):
        pool.copy_on_write(7)                            # never allocated


def test_duplicate_ids_in_one_free_call():
    pool = PoolModel(4)
    (b,) = pool.alloc(1)
    pool.share([b])
    pool.free([b, b])                                    # two references, two releases
    assert pool.ref[b] == 0
    (c,) = pool.alloc(1)
    with pytest.raises(PoolError):
        pool.free([c, c])                                # only one reference
    assert pool.ref[c] == 1


def test_waste_stats_on_the_worked_example(golden):
    """The statistic on the pages' four requests: 25,468 of 32,768 reserved slots
    untouched (77.72 %), 457 paged blocks with 12 slots of internal waste."""
    kv, _ = golden("worked_allocation_example.txt")
    used = [int(x) for x in kv["used_tokens"].split()]
    w = waste_stats(used, int(kv["reservation_tokens"]), int(kv["block_size"]))
    assert w["contiguous_reserved_slots"] == 32768 and w["contiguous_untouched_slots"] == 25468
    assert abs(w["contiguous_untouched_percent"] - 77.72) < 0.01
    assert (w["paged_blocks"], w["paged_waste_slots"]) == (457, 12)
    assert abs(w["paged_waste_percent"] - 100 * 12 / 7312) < 1e-12


def test_waste_stats_closed_forms():
    # block-aligned lengths waste nothing when paged; one token per request wastes 15
    w = waste_stats([16, 32, 4096], 8192)
    assert w["paged_waste_slots"] == 0 and w["paged_blocks"] == 1 + 2 + 256
    w = waste_stats([1] * 10, 16)
    assert w["paged_waste_slots"] == 150 and w["contiguous_untouched_slots"] == 150
    with pytest.raises(PoolError):
        waste_stats([9000], 8192)
