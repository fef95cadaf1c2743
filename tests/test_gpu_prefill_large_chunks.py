"""Chunks whose query rows fill several 128-row tensor-core tiles (chunk tokens
x GQA group >= 512): parity with the fp64 oracle on a chunk of exactly four
tiles, on ragged chunks (a last tile partly past the chunk, computed as padding
and never stored) next to decode rows, over several KV partitions; the tail
of the last block never leaks (NaN-poisoned cache); bitwise identical under
another physical placement."""
import numpy as np
import pytest

import paged_kv_cache_263_gb300 as pkv
from oracle import model as omodel
from paged_kv_cache_263_gb300.workload import DeviceWorkload
from synth.workloads import small_workload
from tests.gpu_util import TOL, check_close, expected_full, max_abs, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    require_gpu()


def _run(wl, poison=False):
    dw = DeviceWorkload(wl, poison_cache=poison)
    dw.step()
    assert pkv.kv_last_device_status() == 0, pkv.kv_last_device_status_flags()
    return dw.out.cpu().numpy().astype(np.float64)


def test_four_full_tiles():
    # 64 tokens x G = 8: four full 128-row tiles, the chunk is the whole context
    wl = small_workload(1500, lens=[64], q_lens=[64], hq=16, hkv=2)
    _, _, ref = expected_full(wl)
    assert max_abs(_run(wl), ref) <= TOL["bf16"]


@pytest.mark.parametrize("hq,hkv", [(16, 2), (32, 8), (32, 2), (64, 8)])
def test_ragged_chunks_next_to_decode_rows(hq, hkv):
    lens = [700, 1, 70, 2100, 33, 129]
    qlens = [100, 1, 70, 300, 1, 65]
    wl = small_workload(1510 + hq, lens=lens, q_lens=qlens, hq=hq, hkv=hkv)
    _, _, ref = expected_full(wl)
    err = max_abs(_run(wl), ref)
    assert err <= TOL["bf16"], err


def test_chunk_over_several_partitions():
    wl = small_workload(1520, lens=[40000, 4000, 17], q_lens=[128, 64, 1], hq=16, hkv=2)
    got = _run(wl)
    cu = wl.cu_q_lens
    for s in range(3):
        check_close(got[cu[s]:cu[s + 1]], omodel.expected_rows(wl, s), "bf16", s)


def test_tail_rows_never_leak():
    lens, qlens = [45, 200, 3001, 77], [45, 70, 100, 1]
    clean = _run(small_workload(1530, lens=lens, q_lens=qlens, hq=16, hkv=2))
    dirty = _run(small_workload(1530, lens=lens, q_lens=qlens, hq=16, hkv=2), poison=True)
    assert np.isfinite(dirty).all()
    assert np.array_equal(clean, dirty)


def test_bitwise_identical_under_block_permutation():
    outs = []
    for perm_seed in (3, 4):
        wl = small_workload(1540, lens=[5000, 300, 12345], q_lens=[256, 1, 200], hq=32, hkv=4)
        wl.free_order = np.random.default_rng(perm_seed).permutation(wl.num_blocks).astype(np.int32)
        outs.append(_run(wl))
    assert np.array_equal(outs[0], outs[1])
