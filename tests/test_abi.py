"""The C-ABI library: it loads without a GPU, exports every symbol the header
declares, and its host block manager agrees bit-exactly with the oracle's
model.  No compute calls are made here."""
import ctypes
import os
import re

import numpy as np
import pytest

import paged_kv_cache_263_gb300 as pkv
from oracle.allocator import PoolError, PoolModel
from paged_kv_cache_263_gb300 import build as pkv_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    pkv_build.build()


def _declared():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            names += re.findall(r"^PAGEDKV_API\s+[^(]*?\b(\w+)\s*\(", src, re.M)
    return names


def test_header_declares_the_boundary():
    names = set(_declared())
    for n in ("kv_block_alloc", "kv_block_free", "kv_block_share", "kv_copy_on_write",
              "reshape_and_cache", "paged_attention_decode", "paged_attention_chunked_prefill"):
        assert n in names


def test_library_exports_every_declared_symbol():
    L = ctypes.CDLL(pkv.library_path)
    for n in _declared():
        assert hasattr(L, n), n


def test_exports_nothing_undeclared():
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", pkv.library_path], capture_output=True,
                         text=True).stdout
    syms = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert syms == set(_declared()), syms ^ set(_declared())


def test_status_strings():
    assert pkv.kv_status_string(0) == "ok"
    assert pkv.kv_status_string(2) == "out of blocks"


def _replay(seed, n_ops=3000, nblocks=300):
    """Random alloc/free/share/cow traffic applied to the library pool and the model."""
    rng = np.random.default_rng(seed)
    order = rng.permutation(nblocks)
    lib_pool = pkv.KVPool(nblocks, order)
    model = PoolModel(nblocks, order)
    owned = []  # list of block ids holding one reference each (owner list)
    for _ in range(n_ops):
        op = rng.integers(0, 5)
        if op == 0:
            n = int(rng.integers(0, 20))
            try:
                got = model.alloc(n)
                ok = True
            except PoolError:
                ok = False
            if ok:
                assert lib_pool.alloc(n).tolist() == got
                owned += got
            else:
                with pytest.raises(pkv.KVError) as e:
                    lib_pool.alloc(n)
                assert e.value.status == 2
        elif op == 1 and owned:
            k = int(rng.integers(1, min(len(owned), 8) + 1))
            idx = rng.choice(len(owned), size=k, replace=False)
            ids = [owned[i] for i in idx]
            for i in sorted(idx, reverse=True):
                owned.pop(i)
            model.free(ids)
            lib_pool.free(ids)
        elif op == 2 and owned:
            ids = [owned[int(rng.integers(len(owned)))] for _ in range(int(rng.integers(1, 4)))]
            model.share(ids)
            lib_pool.share(ids)
            owned += ids
        elif op == 3 and owned:
            i = int(rng.integers(len(owned)))
            b = owned[i]
            try:
                nb, _ = model.copy_on_write(b)
                ok = True
            except PoolError:
                ok = False
            if ok:
                assert lib_pool.copy_on_write(b) == nb
                owned[i] = nb
            else:
                with pytest.raises(pkv.KVError):
                    lib_pool.copy_on_write(b)
        elif op == 4:
            bad = int(rng.integers(0, nblocks))
            if model.ref[bad] == 0:
                with pytest.raises(pkv.KVError) as e:
                    lib_pool.free([bad])
                assert e.value.status == 1
                with pytest.raises(pkv.KVError):
                    lib_pool.share([bad])
        s = lib_pool.stats()
        m = model.stats()
        assert (s["free"], s["live"], s["shared"], s["cow_copies"], s["alloc_failures"]) == \
               (m["free"], m["live"], m["shared"], m["cow_copies"], m["alloc_failures"])
    for b in range(nblocks):
        assert lib_pool.refcount(b) == model.ref[b]
    # the free lists hand out the same blocks in the same order
    rest = model.free_blocks
    assert lib_pool.alloc(rest).tolist() == model.alloc(rest)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_block_manager_matches_model_bit_exactly(seed):
    _replay(seed)


def test_block_tables_of_every_workload_match_the_model():
    from oracle import model as omodel
    from synth.workloads import make_workload
    for name in ("tiny", "llama8b", "llama70b_prefix", "mixed_prefill", "split_fp8"):
        wl = make_workload(name)
        tb = omodel.build_tables(wl)
        pool = pkv.KVPool(wl.num_blocks, wl.free_order)
        B, mb = wl.num_seqs, wl.max_blocks_per_seq
        tables = np.full((B, mb), -1, np.int32)
        pb = -(-wl.prefix_tokens // 16) if wl.prefix_tokens else 0
        if pb:
            pre = pool.alloc(pb)
            tables[0, :pb] = pre
            for s in range(1, B):
                pool.share(pre)
                tables[s, :pb] = pre
        if wl.cow_block >= 0:
            for s in range(B):
                tables[s, wl.cow_block] = pool.copy_on_write(int(tables[s, wl.cow_block]))
        for s in range(B):
            n = -(-int(wl.context_lens[s]) // 16) - pb
            tables[s, pb:pb + n] = pool.alloc(n)
        assert np.array_equal(tables, tb.tables), name
        assert pool.stats()["cow_copies"] == len(tb.copies)


def test_alloc_all_or_nothing_and_fault_injection():
    pool = pkv.KVPool(10)
    pool.alloc(4)
    pool.fail_alloc_after(2)
    pool.alloc(1)                               # first call passes
    before = pool.stats()
    with pytest.raises(pkv.KVError) as e:       # second call is the injected failure
        pool.alloc(1)
    assert e.value.status == 2
    after = pool.stats()
    assert after["free"] == before["free"] and after["alloc_failures"] == before["alloc_failures"] + 1
    pool.alloc(5)                               # disarmed again
    with pytest.raises(pkv.KVError):
        pool.alloc(1)                           # genuinely empty
    # an injected failure inside copy-on-write leaves the pool unchanged
    pool2 = pkv.KVPool(4)
    (b,) = pool2.alloc(1)
    pool2.share([b])
    pool2.fail_alloc_after(1)
    with pytest.raises(pkv.KVError):
        pool2.copy_on_write(b)
    assert pool2.refcount(b) == 2 and pool2.stats()["free"] == 3


def test_pool_rejects_bad_orders():
    with pytest.raises(pkv.KVError):
        pkv.KVPool(3, [0, 0, 1])
    with pytest.raises(pkv.KVError):
        pkv.KVPool(0)


def test_host_validation_before_launch():
    L = pkv.lib()
    # null pointers and bad head ratios are refused without touching a device
    assert L.paged_attention_decode(None, None, None, None, None, 4, None, 1, 8, 2, 64, 0.1, 0, None, None,
                                    0, None, 0, None) == 1
    fake = ctypes.c_void_p(0x10000)
    assert L.paged_attention_decode(fake, fake, fake, fake, fake, 4, fake, 1, 8, 3, 64, 0.1, 0, None, None,
                                    0, None, 0, None) == 1
    assert L.paged_attention_decode(fake, fake, fake, fake, fake, 4, fake, 1, 96, 3, 64, 0.1, 0, None, None,
                                    0, None, 0, None) == 3          # G = 32: unsupported
    assert L.paged_attention_decode(fake, fake, fake, fake, fake, 4, fake, 1, 8, 2, 64, 0.1, 1, None, None,
                                    0, None, 0, None) == 1          # fp8 without scales
    assert L.reshape_and_cache(fake, fake, fake, fake, None, 3, 2, 10, 0, None, None, None) == 1
    assert L.reshape_and_cache(fake, fake, fake, fake, fake, 3, 2, 10, 7, None, None, None) == 3
    # workspace too small for the splits it needs
    need = pkv.paged_attention_workspace_size(2, 8, 100, 4)
    assert need > 0
    assert L.paged_attention_decode(fake, fake, fake, fake, fake, 100, fake, 2, 8, 2, 400, 0.1, 0, None, None,
                                    4, fake, need - 256, None) == 1
    assert pkv.paged_attention_workspace_size(2, 8, 100, 1) == 0
    # fp8 cache with chunks: the scales are required; a short workspace is refused
    assert L.paged_attention_chunked_prefill(fake, fake, fake, fake, 1, 100, 100, fake, fake, fake, 2048, 8, 2,
                                             3000, 0.1, 1, None, None, 0, fake, 1 << 30, None) == 1
    ws = pkv.paged_attention_chunked_prefill_workspace_size(1, 100, 100, 8, 2, 2048, 0)
    assert ws >= 100 * 8 * 2 * 130 * 4          # rows x heads x at least two KV partitions
    assert L.paged_attention_chunked_prefill(fake, fake, fake, fake, 1, 100, 100, fake, fake, fake, 2048, 8, 2,
                                             3000, 0.1, 1, fake, fake, 0, fake, 256, None) == 1


def test_launch_count_follows_the_plan():
    """The kernels a call enqueues, from the host plan alone: decode (+ merge
    when the context is partitioned), short chunks in the multi-row decode
    mode, longer chunks adding the work list, the chunk kernel and its merge --
    and no decode rows when every query is max_q_len long."""
    n = pkv.paged_attention_launch_count
    assert n(0, 0, 1, 8, 2, 100, 0) == 0                  # nothing to do
    assert n(4, 4, 1, 8, 2, 1, 0) == 1                    # one block: one partition, no merge
    assert n(4, 4, 1, 8, 2, 100, 1) == 1                  # one forced partition
    assert n(4, 4, 1, 8, 2, 100, 4) == 2                  # four partitions: merge
    assert n(4, 8, 2, 16, 4, 100, 1) == 1                 # 2 rows x G 4 = 8 columns: multi-row mode
    assert n(4, 8, 2, 16, 4, 100, 4) == 2
    # 4 rows x G 4 = 16 columns: chunk tiles; 4 x 4 rows leave no decode rows
    assert n(4, 16, 4, 16, 4, 60, 1) == 2                 # 960 keys: one partition
    assert n(4, 17, 4, 16, 4, 60, 1) == 1 + 2             # 17 rows: a decode row too
    assert n(4, 20, 5, 16, 4, 60, 1) == 2                 # 5 x 4 columns; 960 keys, one partition
    # a small batch shortens the chunk partitions to 1,024 keys: 1,600 keys take two
    assert n(4, 20, 5, 16, 4, 100, 1) == 3
    assert n(1, 100, 100, 8, 2, 1, 1) == 2                # 16 keys: one partition of the chunk's keys
    # 32,768 keys exceed the longest chunk partition (16,384): the chunk merge runs
    assert n(1, 100, 100, 8, 2, 2048, 1) == 3
    assert n(1, 100, 100, 8, 2, 2048, 4) == 3             # (num_splits is for decode rows: none)
    assert n(2, 101, 100, 8, 2, 2048, 1) == 1 + 3         # a decode row beside the chunk
    assert n(2, 101, 100, 8, 2, 2048, 4) == 2 + 3


def test_bounded_wait_selftest_refuses_bad_limits():
    """The failure-path self-test checks its limit on the host: nothing launches."""
    L = pkv.lib()
    assert L.kv_selftest_bounded_wait(0, None) == 1
    assert L.kv_selftest_bounded_wait(2_000_001, None) == 1


class _FakeDeviceTensor:
    """Stands in for a contiguous CUDA tensor where only the binding's argument
    checks look at it (no GPU here; nothing is launched)."""

    def __init__(self, dtype, shape):
        self.dtype, self.shape, self.is_cuda = dtype, shape, True

    def is_contiguous(self):
        return True


@pytest.mark.parametrize("bad", ["k_cpu", "v_cpu", "k_strided"])
def test_static_scratch_decode_checks_the_caches_before_any_launch(bad, monkeypatch):
    """A CPU or non-contiguous cache is refused by the binding with ValueError
    before the library is called, as paged_attention_decode does."""
    import gc
    import torch

    # records which library entry points are reached (a host object of an
    # earlier test, collected meanwhile, may reach its own destructor's call)
    called = []

    class _Recorder:
        def __getattr__(self, name):
            called.append(name)
            return lambda *a, **k: 0

    gc.collect()
    monkeypatch.setattr(pkv, "lib", lambda: _Recorder())
    out = _FakeDeviceTensor(torch.float32, (2, 8, 128))
    q = _FakeDeviceTensor(torch.bfloat16, (2, 8, 128))
    bt = _FakeDeviceTensor(torch.int32, (2, 4))
    cl = _FakeDeviceTensor(torch.int32, (2,))
    good = _FakeDeviceTensor(torch.bfloat16, (16, 2, 16, 128))
    cpu = torch.zeros(16, 2, 16, 128, dtype=torch.bfloat16)
    k, v = good, good
    if bad == "k_cpu":
        k = cpu
    elif bad == "v_cpu":
        v = cpu
    else:
        k = _FakeDeviceTensor(torch.bfloat16, (16, 2, 16, 128))
        k.is_contiguous = lambda: False
    with pytest.raises(ValueError, match="k_cache|v_cache"):
        pkv.paged_attention_decode_static_scratch(out, q, k, v, bt, cl)
    assert "paged_attention_decode_static_scratch" not in called
