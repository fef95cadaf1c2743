"""GPU parity of the cache write and paged decode against the fp64 oracle.

Tolerances: bf16 cache max-abs 1e-2, fp8 cache 5e-2 (attention outputs);
cache bytes and block tables bit-exact; outputs bitwise identical under any
physical block permutation."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_263_gb300 as pkv
from oracle import model as omodel
from paged_kv_cache_263_gb300.workload import DeviceWorkload
from synth.workloads import make_workload, small_workload
from tests.gpu_util import TOL, bits, cache_bytes, check_close, expected_full, max_abs, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    require_gpu()


# ------------------------------------------------------------- cache write
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_reshape_and_cache_bit_exact(kv_dtype):
    wl = small_workload(101, lens=[37], hq=8, hkv=4, kv_dtype=kv_dtype, num_blocks=40)
    T = 77
    keys = np.arange(1000, 1000 + T)
    k = wl.kv_values("k", keys)
    v = wl.kv_values("v", keys)
    rng = np.random.default_rng(5)
    slots = rng.choice(40 * 16, size=T, replace=False).astype(np.int64)
    slots[[3, 40, 76]] = -1                       # padding tokens are skipped
    if kv_dtype == "fp8":
        ks = np.array([0.004, 0.01, 0.02, 0.5], np.float32)   # head 0 saturates (x/s up to ~870)
        vs = np.array([0.0077, 0.2, 0.003, 1.0], np.float32)
    else:
        ks = vs = None
    shape = (40, 4, 16, 128)
    ref_k = np.zeros(shape, np.uint8 if kv_dtype == "fp8" else np.uint16)
    ref_v = np.zeros_like(ref_k)
    oracle.reshape_and_cache(bits(k), bits(v), ref_k, ref_v, slots,
                             oracle.FP8 if kv_dtype == "fp8" else oracle.BF16, ks, vs)
    cdt = torch.uint8 if kv_dtype == "fp8" else torch.bfloat16
    kc = torch.zeros(shape, dtype=cdt, device="cuda")
    vc = torch.zeros(shape, dtype=cdt, device="cuda")
    pkv.reshape_and_cache(k.cuda(), v.cuda(), kc, vc, torch.from_numpy(slots).cuda(),
                          None if ks is None else torch.from_numpy(ks).cuda(),
                          None if vs is None else torch.from_numpy(vs).cuda())
    assert pkv.kv_last_device_status() == 0
    assert np.array_equal(cache_bytes(kc), ref_k)
    assert np.array_equal(cache_bytes(vc), ref_v)


def test_reshape_and_cache_flags_slot_outside_pool():
    k = torch.ones(3, 2, 128, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(4, 2, 16, 128, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    slots = torch.tensor([1, 4 * 16 + 3, 63], dtype=torch.int64, device="cuda")
    pkv.reshape_and_cache(k, k, kc, vc, slots)
    assert pkv.kv_last_device_status() == 5
    assert pkv.kv_last_device_status_flags() & 2
    assert kc[0, :, 1].float().eq(1).all() and kc[3, :, 15].float().eq(1).all()
    assert kc.float().sum().item() == 2 * 2 * 128
    assert pkv.kv_last_device_status() == 0       # cleared


# ----------------------------------------------------------- decode parity
def _run(wl, poison=False):
    dw = DeviceWorkload(wl, poison_cache=poison)
    dw.step()
    assert pkv.kv_last_device_status() == 0
    return dw, dw.out.cpu().numpy().astype(np.float64)


def test_tiny_config_matches_oracle():
    wl = make_workload("tiny")
    tb, caches, ref = expected_full(wl)
    dw, got = _run(wl)
    assert np.array_equal(dw.tables_host, tb.tables)
    assert np.array_equal(cache_bytes(dw.k_cache), caches[0])
    assert np.array_equal(cache_bytes(dw.v_cache), caches[1])
    assert max_abs(got, ref) <= TOL["bf16"]


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 4), (8, 2), (16, 2), (32, 2)])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_decode_small_cases(kv_dtype, hq, hkv, splits):
    lens = [1, 15, 16, 17, 33, 130, 700, 1201]
    wl = small_workload(200 + hq + hkv, lens=lens, hq=hq, hkv=hkv, kv_dtype=kv_dtype)
    wl.num_splits = splits
    _, _, ref = expected_full(wl)
    _, got = _run(wl)
    err = max_abs(got, ref)
    assert err <= TOL[kv_dtype], err


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_bitwise_identical_under_block_permutation(kv_dtype):
    lens = [5, 64, 129, 999, 2048]
    outs = []
    for perm_seed in (1, 2, 3):
        wl = small_workload(300, lens=lens, hq=16, hkv=2, kv_dtype=kv_dtype, num_splits=4)
        wl.free_order = np.random.default_rng(perm_seed).permutation(wl.num_blocks).astype(np.int32)
        outs.append(_run(wl)[1])
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_unwritten_slots_never_leak():
    """The cache is filled with NaN before the workload is written; the tail of
    the last block (never written) must not reach the output."""
    wl = small_workload(400, lens=[3, 17, 50, 333], hq=8, hkv=2)
    _, clean = _run(wl)
    wl2 = small_workload(400, lens=[3, 17, 50, 333], hq=8, hkv=2)
    _, dirty = _run(wl2, poison=True)
    assert np.isfinite(dirty).all()
    assert np.array_equal(clean, dirty)


def test_bad_block_id_and_length_are_flagged_not_faulted():
    wl = small_workload(500, lens=[40, 40], hq=8, hkv=2)
    dw = DeviceWorkload(wl)
    dw.block_tables[1, 1] = wl.num_blocks + 7          # outside the pool
    dw.attention()
    assert pkv.kv_last_device_status() == 5
    assert pkv.kv_last_device_status_flags() & 1
    dw.block_tables[1, 1] = int(dw.tables_host[1, 1])
    dw.context_lens[0] = wl.max_blocks_per_seq * 16 + 1  # longer than its table row
    dw.attention()
    assert pkv.kv_last_device_status() == 5
    assert pkv.kv_last_device_status_flags() & 4
    assert (dw.out[0] == 0).all()


def test_copy_on_write_device_copy():
    wl = small_workload(600, lens=[40, 45], hq=8, hkv=2, prefix_tokens=40, cow_block=2)
    dw = DeviceWorkload(wl)
    tb, caches, ref = expected_full(wl)
    assert np.array_equal(dw.tables_host, tb.tables)
    assert dw.pool.stats()["cow_copies"] == 1
    dw.step()                                   # writes the step's new tokens too
    assert pkv.kv_last_device_status() == 0
    assert np.array_equal(cache_bytes(dw.k_cache), caches[0])
    assert np.array_equal(cache_bytes(dw.v_cache), caches[1])
    assert max_abs(dw.out.cpu().numpy(), ref) <= TOL["bf16"]


def test_empty_batches_launch_nothing_and_succeed():
    """Zero tokens to write, zero sequences to decode, a mixed batch with no query
    rows and one whose sequences contribute none: each call returns success, the
    cache is untouched and no device flag is raised."""
    dev = "cuda"
    kc = torch.full((4, 2, 16, 128), 0.5, dtype=torch.bfloat16, device=dev)
    vc = kc.clone()
    before = kc.clone()
    e = torch.empty(0, 2, 128, dtype=torch.bfloat16, device=dev)
    pkv.reshape_and_cache(e, e, kc, vc, torch.empty(0, dtype=torch.int64, device=dev))
    out = torch.empty(0, 8, 128, dtype=torch.float32, device=dev)
    q = torch.empty(0, 8, 128, dtype=torch.bfloat16, device=dev)
    bt = torch.zeros(0, 4, dtype=torch.int32, device=dev)
    cl = torch.zeros(0, dtype=torch.int32, device=dev)
    pkv.paged_attention_decode(out, q, kc, vc, bt, cl)
    pkv.paged_attention_chunked_prefill(out, q, torch.zeros(1, dtype=torch.int32, device=dev), cl, 1, kc, vc, bt)
    # two sequences with context but no query rows this step
    bt2 = torch.tensor([[0, 1, -1, -1], [2, -1, -1, -1]], dtype=torch.int32, device=dev)
    cl2 = torch.tensor([20, 9], dtype=torch.int32, device=dev)
    cu2 = torch.zeros(3, dtype=torch.int32, device=dev)
    pkv.paged_attention_chunked_prefill(out, q, cu2, cl2, 1, kc, vc, bt2)
    torch.cuda.synchronize()
    assert pkv.kv_last_device_status() == 0
    assert torch.equal(kc, before) and torch.equal(vc, before)


def test_million_token_context_over_many_partitions():
    """A 2^20-token context (65,536 blocks): 256 split-KV partitions merged in one
    log-sum-exp pass, next to a short sequence; both against the oracle."""
    wl = small_workload(1700, lens=[1 << 20, 777], hq=8, hkv=2)
    dw, got = _run(wl)
    for s in range(2):
        check_close(got[s:s + 1], omodel.expected_rows(wl, s), "bf16", s)
