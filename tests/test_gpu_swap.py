"""Swap-out / swap-in on the GPU: bytes bit-exact against the oracle's gather
and scatter, ids outside the pool skipped and flagged, and a preempted
sequence brought back into other physical blocks attends bitwise as before."""
import numpy as np
import pytest
import torch

import paged_kv_cache_263_gb300 as pkv
from oracle.swap import swap_in as o_swap_in, swap_out as o_swap_out
from paged_kv_cache_263_gb300.workload import DeviceWorkload
from synth.workloads import small_workload
from tests.gpu_util import cache_bytes, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    require_gpu()


def _random_cache(nb, hkv, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    if dtype == torch.bfloat16:
        x = torch.randint(-32768, 32768, (nb, hkv, 16, 128), dtype=torch.int32, generator=g).to(torch.int16)
        return x.view(torch.bfloat16).cuda()
    return torch.randint(0, 256, (nb, hkv, 16, 128), dtype=torch.int32, generator=g).to(torch.uint8).cuda()


def _pinned(n, like):
    return torch.empty((n,) + tuple(like.shape[1:]), dtype=like.dtype).pin_memory()


@pytest.mark.parametrize("dtype,hkv,n", [(torch.bfloat16, 8, 300), (torch.uint8, 8, 257), (torch.bfloat16, 1, 3)])
def test_swap_out_and_in_are_bit_exact(dtype, hkv, n):
    nb = 1000
    k, v = _random_cache(nb, hkv, dtype, 1), _random_cache(nb, hkv, dtype, 2)
    rng = np.random.default_rng(n)
    ids = rng.choice(nb, size=n, replace=False).astype(np.int32)
    ids[-1] = ids[0] if n > 2 else ids[-1]               # a repeat is fine for swap-out
    hk, hv = _pinned(n, k), _pinned(n, v)
    pkv.kv_swap_out(k, v, torch.from_numpy(ids).cuda(), hk, hv)
    torch.cuda.synchronize()
    assert pkv.kv_last_device_status() == 0
    ek, ev = o_swap_out(cache_bytes(k), cache_bytes(v), ids)
    assert np.array_equal(cache_bytes(hk), ek) and np.array_equal(cache_bytes(hv), ev)
    # back into other, distinct blocks of a fresh cache
    new = rng.choice(nb, size=n, replace=False).astype(np.int32)
    k2, v2 = _random_cache(nb, hkv, dtype, 3), _random_cache(nb, hkv, dtype, 4)
    want_k, want_v = cache_bytes(k2).copy(), cache_bytes(v2).copy()
    pkv.kv_swap_in(k2, v2, torch.from_numpy(new).cuda(), hk, hv)
    torch.cuda.synchronize()
    assert pkv.kv_last_device_status() == 0
    o_swap_in(want_k, want_v, new, ek, ev)
    assert np.array_equal(cache_bytes(k2), want_k) and np.array_equal(cache_bytes(v2), want_v)


def test_ids_outside_the_pool_are_skipped_and_flagged():
    nb = 16
    k, v = _random_cache(nb, 2, torch.bfloat16, 5), _random_cache(nb, 2, torch.bfloat16, 6)
    ids = torch.tensor([3, nb, -1, 7], dtype=torch.int32, device="cuda")
    hk, hv = _pinned(4, k), _pinned(4, v)
    hk.view(torch.int16).fill_(0x1234)
    hv.view(torch.int16).fill_(0x1234)
    pkv.kv_swap_out(k, v, ids, hk, hv)
    assert pkv.kv_last_device_status() == 5 and pkv.kv_last_device_status_flags() & 1
    kb = cache_bytes(k)
    got = cache_bytes(hk)
    assert np.array_equal(got[0], kb[3]) and np.array_equal(got[3], kb[7])
    assert (got[1] == 0x1234).all() and (got[2] == 0x1234).all()


def test_non_pinned_host_memory_is_refused():
    k = _random_cache(4, 1, torch.bfloat16, 7)
    ids = torch.tensor([0], dtype=torch.int32, device="cuda")
    hk = torch.empty((1, 1, 16, 128), dtype=torch.bfloat16)      # pageable
    st = pkv.lib().kv_swap_out(k.data_ptr(), k.data_ptr(), 4, 1, 0, ids.data_ptr(), 1, hk.data_ptr(),
                               hk.data_ptr(), None)
    assert st == 1


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_preempted_sequence_comes_back_bitwise(kv_dtype):
    """Sequence 1 is swapped out, its blocks are reused (overwritten), and it is
    swapped back into other free blocks with its table row rewritten: every
    sequence's output is bitwise unchanged."""
    wl = small_workload(31, lens=[300, 2000, 77, 4100], hq=16, hkv=2, kv_dtype=kv_dtype, num_blocks=1200)
    dw = DeviceWorkload(wl)
    dw.step()
    before = dw.out.clone()
    row = dw.tables_host[1]
    old = row[row >= 0]
    pool = dw.pool
    old_dev = torch.from_numpy(old.astype(np.int32)).cuda()
    hk, hv = _pinned(len(old), dw.k_cache), _pinned(len(old), dw.v_cache)
    pkv.kv_swap_out(dw.k_cache, dw.v_cache, old_dev, hk, hv)
    torch.cuda.synchronize()
    pool.free(old)                                      # preempted: its blocks go back to the pool
    junk = pool.alloc(len(old))                         # another request takes them and writes
    jd = torch.from_numpy(junk.astype(np.int64)).cuda()
    dw.k_cache[jd] = dw.k_cache[jd].flip(-1)
    dw.v_cache[jd] = dw.v_cache[jd].flip(-2)
    new = pool.alloc(len(old))                          # resumed: wherever the pool has room
    assert not set(new.tolist()) & set(old.tolist())
    pkv.kv_swap_in(dw.k_cache, dw.v_cache, torch.from_numpy(new.astype(np.int32)).cuda(), hk, hv)
    dw.block_tables[1, :len(new)] = torch.from_numpy(new.astype(np.int32)).cuda()
    dw.attention()
    assert pkv.kv_last_device_status() == 0
    assert torch.equal(before, dw.out)
