"""GPU parity of the mixed chunked-prefill / decode call against the fp64 oracle
(max-abs 1e-2 for the bf16 cache, 5e-2 for fp8), bitwise permutation
invariance, and the full-size mixed workload on sampled rows."""
import numpy as np
import pytest

import paged_kv_cache_263_gb300 as pkv
from oracle import model as omodel
from paged_kv_cache_263_gb300.workload import DeviceWorkload
from synth.workloads import make_workload, small_workload
from tests.gpu_util import TOL, check_close, expected_full, max_abs, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    require_gpu()


def _run(wl, poison=False):
    dw = DeviceWorkload(wl, poison_cache=poison)
    dw.step()
    assert pkv.kv_last_device_status() == 0, pkv.kv_last_device_status_flags()
    return dw, dw.out.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 4), (8, 2), (16, 2), (32, 2)])
def test_mixed_batch_small(hq, hkv):
    lens = [1, 2, 20, 300, 64, 700, 129]
    qlens = [1, 2, 17, 1, 64, 130, 129]          # a chunk equal to its whole context, too
    wl = small_workload(700 + hq, lens=lens, q_lens=qlens, hq=hq, hkv=hkv)
    _, _, ref = expected_full(wl)
    _, got = _run(wl)
    err = max_abs(got, ref)
    assert err <= TOL["bf16"], err


def test_chunk_spanning_several_partitions():
    """A 40-row chunk over 40,000 keys: several KV partitions merged by LSE."""
    wl = small_workload(800, lens=[40000, 33], q_lens=[40, 1], hq=16, hkv=2)
    _, got = _run(wl)
    cu = wl.cu_q_lens
    for s in range(2):
        check_close(got[cu[s]:cu[s + 1]], omodel.expected_rows(wl, s), "bf16", s)


def test_prefill_bitwise_identical_under_block_permutation():
    outs = []
    for perm_seed in (1, 2):
        wl = small_workload(900, lens=[500, 37, 20000], q_lens=[130, 1, 77], hq=8, hkv=1)
        wl.free_order = np.random.default_rng(perm_seed).permutation(wl.num_blocks).astype(np.int32)
        outs.append(_run(wl)[1])
    assert np.array_equal(outs[0], outs[1])


def test_prefill_unwritten_slots_never_leak():
    wl = small_workload(950, lens=[45, 200], q_lens=[45, 9], hq=8, hkv=2)
    _, clean = _run(wl)
    wl2 = small_workload(950, lens=[45, 200], q_lens=[45, 9], hq=8, hkv=2)
    _, dirty = _run(wl2, poison=True)
    assert np.isfinite(dirty).all()
    assert np.array_equal(clean, dirty)


@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 2), (16, 2), (32, 2)])
def test_fp8_mixed_batch_small(hq, hkv):
    """fp8 cache with chunks: every row is its own decode problem over keys 0 .. L-n+i."""
    lens = [1, 2, 20, 300, 64, 700, 129]
    qlens = [1, 2, 17, 1, 64, 130, 129]
    wl = small_workload(960 + hq, lens=lens, q_lens=qlens, hq=hq, hkv=hkv, kv_dtype="fp8")
    _, _, ref = expected_full(wl)
    _, got = _run(wl)
    err = max_abs(got, ref)
    assert err <= TOL["fp8"], err


def test_fp8_chunk_spanning_several_partitions():
    wl = small_workload(970, lens=[40000, 33], q_lens=[40, 1], hq=16, hkv=2, kv_dtype="fp8")
    _, got = _run(wl)
    cu = wl.cu_q_lens
    for s in range(2):
        err = max_abs(got[cu[s]:cu[s + 1]], omodel.expected_rows(wl, s))
        assert err <= TOL["fp8"], (s, err)


def test_fp8_chunks_bitwise_identical_under_block_permutation_and_poison():
    outs = []
    for perm_seed, poison in ((1, False), (2, True)):
        wl = small_workload(980, lens=[500, 37, 20000], q_lens=[130, 1, 77], hq=8, hkv=1, kv_dtype="fp8")
        wl.free_order = np.random.default_rng(perm_seed).permutation(wl.num_blocks).astype(np.int32)
        outs.append(_run(wl, poison=poison)[1])
    assert np.isfinite(outs[1]).all()
    assert np.array_equal(outs[0], outs[1])


def test_mixed_prefill_workload_sampled():
    wl = make_workload("mixed_prefill")
    tb = omodel.build_tables(wl)
    dw = DeviceWorkload(wl)
    assert np.array_equal(dw.tables_host, tb.tables)
    dw.step()
    assert pkv.kv_last_device_status() == 0
    out = dw.out.cpu().numpy()
    cu = wl.cu_q_lens
    rows = [0, 1, 15, 16, 17, 511, 1000, 1023]
    ref = omodel.expected_rows(wl, 0, rows=rows)
    check_close(out[cu[0] + np.array(rows)], ref, "bf16", "chunk")
    for s in (1, 100, 255):
        check_close(out[cu[s]:cu[s + 1]], omodel.expected_rows(wl, s), "bf16", s)


@pytest.mark.parametrize("hq,hkv,n,dt", [(32, 8, 4, "bf16"), (64, 8, 8, "bf16"), (16, 2, 6, "bf16"),
                                         (8, 8, 5, "bf16"), (16, 1, 4, "bf16"), (32, 8, 4, "fp8"),
                                         (64, 8, 8, "fp8")])
def test_spec_verify_shapes_small(hq, hkv, n, dt):
    """Speculative verification: every sequence checks an n-token draft, n causal
    rows each ("M.65 Inference serving", speculative decoding, N = 4-8).  Up to
    8 columns (rows x G) the chunks run in the decode kernel's multi-row mode,
    beyond that in the tensor-core kernel; a 17-token context with a 4-row
    chunk leaves some rows no visible key in the last block."""
    lens = [n, 40, 300, 1025, 16, 17, 4096]
    qlens = [n] * len(lens)
    qlens[1] = 1                                  # a decode row in the same batch
    wl = small_workload(1100 + n, lens=lens, q_lens=qlens, hq=hq, hkv=hkv, kv_dtype=dt)
    _, _, ref = expected_full(wl)
    _, got = _run(wl)
    assert max_abs(got, ref) <= TOL[dt]


@pytest.mark.parametrize("name", ["spec_verify", "spec_verify8"])
def test_spec_verify_workloads_sampled(name):
    wl = make_workload(name)
    _, out = _run(wl)
    cu = wl.cu_q_lens
    for s in (0, 1, wl.num_seqs // 2, wl.num_seqs - 1):
        check_close(out[cu[s]:cu[s + 1]], omodel.expected_rows(wl, s), "bf16", s)


def test_calls_from_several_streams_and_a_captured_graph():
    """The mixed call issued from a second stream, captured into a CUDA graph and
    replayed, then eagerly again from the default stream: every call completes
    within its time limits (status 0) and gives bitwise the same output."""
    import torch
    wl = make_workload("spec_verify8")
    dw = DeviceWorkload(wl)
    dw.step()
    assert pkv.kv_last_device_status() == 0
    ref = dw.out.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            dw.attention()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        dw.attention()
    for _ in range(20):
        g.replay()
    torch.cuda.synchronize()
    assert pkv.kv_last_device_status() == 0
    assert torch.equal(dw.out, ref)
    for _ in range(60):
        dw.attention()
    assert pkv.kv_last_device_status() == 0, pkv.kv_last_device_status_flags()
    assert torch.equal(dw.out, ref)


@pytest.mark.parametrize("qlens,dt", [([5, 0, 1, 0], "bf16"), ([4, 0, 1, 0], "bf16"), ([4, 0, 1, 0], "fp8"),
                                      ([40, 0, 1, 0], "fp8"), ([2, 0, 1, 0], "bf16"), ([2, 0, 1, 0], "fp8")])
def test_sequences_with_no_query_rows(qlens, dt):
    """A sequence may contribute no rows to a mixed batch (cu_q_lens repeats a
    value): the tensor-core path (5 or 4 rows x G 4, and 40 rows over an fp8
    cache) and the multi-row mode (2 x 4) all skip it and get every other row
    right."""
    wl = small_workload(1200 + sum(qlens), lens=[100, 50, 300, 17], q_lens=qlens, hq=16, hkv=4, kv_dtype=dt)
    _, _, ref = expected_full(wl)
    _, got = _run(wl)
    assert got.shape == ref.shape
    assert max_abs(got, ref) <= TOL[dt]


def test_mixed_prefill_fp8_workload_sampled():
    """The mixed batch over an fp8 cache: the 1,024-row chunk runs on the tensor
    cores with e4m3 K/V widened to f16 operands."""
    wl = make_workload("mixed_prefill_fp8")
    dw = DeviceWorkload(wl)
    dw.step()
    assert pkv.kv_last_device_status() == 0
    out = dw.out.cpu().numpy()
    cu = wl.cu_q_lens
    rows = [0, 1, 15, 16, 17, 511, 1000, 1023]
    ref = omodel.expected_rows(wl, 0, rows=rows)
    check_close(out[cu[0] + np.array(rows)], ref, "fp8", "chunk")
    for s in (1, 100, 255):
        check_close(out[cu[s]:cu[s + 1]], omodel.expected_rows(wl, s), "fp8", s)


def test_chunk_kernel_trace_events():
    wl = small_workload(1500, lens=[3000, 40], q_lens=[256, 1], hq=16, hkv=2)
    dw = DeviceWorkload(wl)
    dw.step()
    pkv.kv_trace_prefill(True)
    dw.attention()
    ms = pkv.kv_trace_prefill_kernel_ms()
    assert 0 < ms < 1000
    assert pkv.kv_trace_prefill_kernel_ms() < 0          # consumed
    pkv.kv_trace_prefill(False)
    dw.attention()
    assert pkv.kv_trace_prefill_kernel_ms() < 0          # not recorded while disabled
    assert pkv.kv_last_device_status() == 0


@pytest.mark.parametrize("hq,hkv,qlens", [(32, 4, [8, 9, 16]), (16, 8, [64, 3, 1]), (8, 2, [32, 32, 1])])
def test_one_tile_chunks_never_leak_and_match(hq, hkv, qlens):
    """Chunks whose rows x heads fit one 128-row tile (the second tile of the
    CTA absent): parity with the oracle, and a NaN-poisoned cache gives the
    same bits."""
    lens = [80, 200, 3001]
    wl = small_workload(1600 + hq, lens=lens, q_lens=qlens, hq=hq, hkv=hkv)
    _, _, ref = expected_full(wl)
    _, clean = _run(wl)
    assert max_abs(clean, ref) <= TOL["bf16"]
    _, dirty = _run(small_workload(1600 + hq, lens=lens, q_lens=qlens, hq=hq, hkv=hkv), poison=True)
    assert np.isfinite(dirty).all() and np.array_equal(clean, dirty)


def test_one_tile_chunk_over_many_partitions():
    wl = small_workload(1610, lens=[40000, 7000, 33], q_lens=[16, 10, 1], hq=64, hkv=8)
    _, got = _run(wl)
    cu = wl.cu_q_lens
    for s in range(3):
        assert max_abs(got[cu[s]:cu[s + 1]], omodel.expected_rows(wl, s)) <= TOL["bf16"], s


@pytest.mark.parametrize("qlens,max_q_len", [([1, 5], 3), ([2, 5, 2], 3), ([1, 3, 2], 2)])
def test_queries_outside_the_declared_bound_are_flagged(qlens, max_q_len):
    """max_q_len bounds every query.  When total_q_tokens = num_seqs x max_q_len
    the chunk path runs no decode rows, so a 1-row query there breaks the
    contract; so does a query longer than max_q_len (in the multi-row decode
    mode -- max_q_len x G <= 8, the last case -- one whose columns exceed the
    CTA's).  Each is flagged as out of range (status 5) and left out, and the
    rows of the queries within the bound still match the oracle."""
    wl = small_workload(1300 + sum(qlens), lens=[60, 300, 90][:len(qlens)], q_lens=qlens, hq=16, hkv=4)
    assert max_q_len * 4 <= 8 or int(wl.q_lens.sum()) == len(qlens) * max_q_len
    dw = DeviceWorkload(wl)
    dw.step()
    pkv.kv_last_device_status()                    # the step's own call used the true maximum: clean
    dw.out.fill_(0.0)
    pkv.paged_attention_chunked_prefill(dw.out, dw.q, dw.cu_q_lens, dw.context_lens, max_q_len, dw.k_cache,
                                        dw.v_cache, dw.block_tables)
    assert pkv.kv_last_device_status() == 5
    assert pkv.kv_last_device_status_flags() & 4   # ST_BAD_LEN
    got = dw.out.cpu().numpy().astype(np.float64)
    cu = wl.cu_q_lens
    multi = max_q_len * 4 <= 8
    for s, n in enumerate(qlens):
        if (1 if multi else 2) <= n <= max_q_len:
            check_close(got[cu[s]:cu[s + 1]], omodel.expected_rows(wl, s), "bf16", s)


def test_large_batches_take_the_global_memory_paths():
    """9,000 sequences, each verifying a 2-token draft (16 columns at G = 8: the
    tensor-core kernel, one query item per sequence): more sequences than the
    work-list kernel stages in shared memory (2,048) and more query items than
    it tables (8,192), so it reads the chunk metadata and searches the item
    prefix sums in global memory; every row still matches the oracle."""
    rng = np.random.default_rng(1400)
    lens = rng.integers(16, 120, size=9000).astype(np.int32)
    wl = small_workload(1400, lens=lens, q_lens=np.full(9000, 2, np.int32), hq=16, hkv=2)
    _, _, ref = expected_full(wl)
    _, got = _run(wl)
    check_close(got, ref, "bf16", "9,000 sequences")


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_many_ragged_chunks_in_the_pair_layout(kv_dtype):
    """48 sequences with 40-row chunks over contexts of 300..6,000 keys.  With
    G = 8 a chunk's rows x heads fill three 128-row tiles, so it takes the
    64-key layout as one item of two query tiles and one item of a single tile
    (the second issuer idle); the work-list kernel orders the ragged items
    longest first and may leave their key ranges whole.  Every row matches the
    oracle."""
    rng = np.random.default_rng(1500)
    lens = rng.integers(300, 6000, size=48).astype(np.int32)
    wl = small_workload(1500, lens=lens, q_lens=np.full(48, 40, np.int32), hq=16, hkv=2, kv_dtype=kv_dtype)
    _, _, ref = expected_full(wl)
    _, got = _run(wl)
    check_close(got, ref, kv_dtype, "48 ragged chunks")


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_decode_heavy_mixed_batch(kv_dtype):
    """One 32-row chunk over 16,384 keys (cut into partitions and merged) beside
    100 decode rows of 200..700 keys: the decode rows' bytes outweigh the chunk's
    work, so the work-list kernel leaves many SMs without a chunk CTA and the
    decode kernel, launched right behind the chunk kernel, runs there.  Every
    row matches the oracle, and a NaN-poisoned pool gives the same bits."""
    rng = np.random.default_rng(1700)
    lens = np.concatenate([[16384], rng.integers(200, 700, size=100)]).astype(np.int32)
    qlens = np.concatenate([[32], np.ones(100, np.int32)]).astype(np.int32)
    wl = small_workload(1700, lens=lens, q_lens=qlens, hq=16, hkv=4, kv_dtype=kv_dtype)
    _, _, ref = expected_full(wl)
    _, got = _run(wl)
    check_close(got, ref, kv_dtype, "decode-heavy mixed batch")
    _, dirty = _run(small_workload(1700, lens=lens, q_lens=qlens, hq=16, hkv=4, kv_dtype=kv_dtype), poison=True)
    assert np.array_equal(got, dirty)
