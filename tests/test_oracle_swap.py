"""Pins of the swap model: element-by-element loops on tiny pools, and the
round trip through other physical blocks leaving paged attention unchanged."""
import numpy as np
import pytest

import oracle
from oracle.swap import swap_in, swap_out


def _cache(rng, nb, hkv, dtype):
    if dtype == np.uint16:
        return rng.integers(0, 1 << 16, size=(nb, hkv, 16, 128), dtype=np.uint16)
    return rng.integers(0, 256, size=(nb, hkv, 16, 128), dtype=np.uint8)


@pytest.mark.parametrize("dtype", [np.uint16, np.uint8])
def test_swap_out_is_the_listed_tiles_in_order(dtype):
    rng = np.random.default_rng(1)
    k, v = _cache(rng, 9, 2, dtype), _cache(rng, 9, 2, dtype)
    ids = [7, 0, 3, 3, 8]
    hk, hv = swap_out(k, v, ids)
    assert hk.shape == (5, 2, 16, 128)
    for i, b in enumerate(ids):
        for h in range(2):
            for t in range(16):
                assert (hk[i, h, t] == k[b, h, t]).all() and (hv[i, h, t] == v[b, h, t]).all()
    with pytest.raises(IndexError):
        swap_out(k, v, [9])


def test_swap_in_writes_only_the_listed_blocks():
    rng = np.random.default_rng(2)
    k, v = _cache(rng, 6, 1, np.uint16), _cache(rng, 6, 1, np.uint16)
    k0, v0 = k.copy(), v.copy()
    hk, hv = _cache(rng, 2, 1, np.uint16), _cache(rng, 2, 1, np.uint16)
    swap_in(k, v, [4, 1], hk, hv)
    for b in range(6):
        if b in (4, 1):
            i = [4, 1].index(b)
            assert (k[b] == hk[i]).all() and (v[b] == hv[i]).all()
        else:
            assert (k[b] == k0[b]).all() and (v[b] == v0[b]).all()
    with pytest.raises(ValueError):
        swap_in(k, v, [2, 2], hk, hv)


def test_round_trip_through_other_blocks_keeps_attention_bitwise():
    """A sequence swapped out and back into other physical blocks, with its
    block table rewritten, gives bitwise the same fp64 oracle output."""
    rng = np.random.default_rng(3)
    nb, hkv, hq, L = 20, 2, 4, 70
    k = rng.integers(0, 1 << 16, size=(nb, hkv, 16, 128), dtype=np.uint16) & 0x3FFF   # finite bf16
    v = rng.integers(0, 1 << 16, size=(nb, hkv, 16, 128), dtype=np.uint16) & 0x3FFF
    q = rng.integers(0, 1 << 16, size=(1, hq, 128), dtype=np.uint16) & 0x3FFF
    table = np.array([[3, 11, 0, 17, 6]], dtype=np.int32)
    before = oracle.paged_attention(q, k, v, table, [L])
    hk, hv = swap_out(k, v, table[0])
    new = np.array([[19, 2, 8, 5, 13]], dtype=np.int32)
    k2 = np.zeros_like(k)
    v2 = np.zeros_like(v)
    swap_in(k2, v2, new[0], hk, hv)
    after = oracle.paged_attention(q, k2, v2, new, [L])
    assert np.array_equal(before, after)
