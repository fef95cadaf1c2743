"""The decode entry point for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc where they run attention (code inside an
allocator or memory-pool hook, a serving runtime that forbids allocation once
it is up, a host without any allocator), so they cannot hand the library the
workspace its split-KV partials need.  paged_attention_decode_static_scratch
keeps those partials in a fixed-size device array inside the library instead.
Here it is called through the C ABI twice in a row, on two different batches
that both need split partials.  Each output must equal, bit for bit, the output
of the ordinary paged_attention_decode (caller workspace) on the same inputs --
the two run the same kernels with the same partitions, only the partials live
elsewhere -- and must match the fp64 oracle within the parity tolerance.
The file name sorts last so a stop-at-first-failure run has already run every
other test when it gets here."""
import numpy as np
import pytest
import torch

import paged_kv_cache_263_gb300 as pkv
from paged_kv_cache_263_gb300.workload import DeviceWorkload
from oracle import model as omodel
from synth.workloads import make_workload, small_workload
from tests.gpu_util import TOL, expected_full, max_abs, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    require_gpu()


def _both(dw):
    wl = dw.wl
    dw.step()
    ref = dw.out.clone()
    got = torch.full_like(dw.out, float("nan"))
    pkv.paged_attention_decode_static_scratch(got, dw.q, dw.k_cache, dw.v_cache, dw.block_tables,
                                              dw.context_lens, wl.scale, dw.k_scale, dw.v_scale,
                                              wl.num_splits)
    assert pkv.kv_last_device_status() == 0
    return ref.cpu().numpy(), got.cpu().numpy()


def test_static_scratch_decode_matches_workspace_decode_twice():
    cap = pkv.paged_attention_decode_static_scratch_bytes()
    first = DeviceWorkload(make_workload("llama8b"))
    wl2 = small_workload(77, lens=[5, 900, 3000, 17, 2500], hq=32, hkv=8, kv_dtype="fp8", num_splits=7)
    second = DeviceWorkload(wl2)
    for dw in (first, second):
        wl = dw.wl
        need = pkv.paged_attention_workspace_size(wl.num_seqs, wl.num_q_heads, wl.max_blocks_per_seq,
                                                  wl.num_splits)
        assert 0 < need <= cap                 # both calls really use the scratch
        ref, got = _both(dw)
        assert np.isfinite(got).all()
        assert np.array_equal(got, ref)
        if wl.num_seqs > 8:
            # the large batch: the oracle's rows of the shortest, longest and two more sequences
            order = np.argsort(wl.context_lens)
            seqs = [int(order[0]), int(order[-1]), 7, 40]
            for s in seqs:
                assert max_abs(got[s:s + 1], omodel.expected_rows(wl, s)) <= TOL[wl.kv_dtype]
        else:
            _, _, exp = expected_full(wl)
            assert max_abs(got, exp) <= TOL[wl.kv_dtype]


def test_static_scratch_refuses_batches_that_do_not_fit():
    wl = small_workload(78, lens=[40, 40], hq=8, hkv=2)
    dw = DeviceWorkload(wl)
    cap = pkv.paged_attention_decode_static_scratch_bytes()
    # a table row long enough that the partials of 2 sequences x 8 heads exceed the array
    splits = 8192
    need = pkv.paged_attention_workspace_size(2, 8, splits, splits)
    assert need > cap
    wide = torch.zeros(2, splits, dtype=torch.int32, device="cuda")
    wide[:, :dw.block_tables.shape[1]] = dw.block_tables
    with pytest.raises(pkv.KVError) as e:
        pkv.paged_attention_decode_static_scratch(dw.out, dw.q, dw.k_cache, dw.v_cache, wide,
                                                  dw.context_lens, wl.scale, num_splits=splits)
    assert e.value.status == 3
