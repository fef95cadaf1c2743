"""Parallel sampling on the GPU: n samples of one prompt share its blocks, the
partial block is copied on each sample's first write (kv_copy_on_write's
device copy), and each sample's decode step -- or its speculative draft
verification -- matches the fp64 oracle."""
import numpy as np
import pytest

import paged_kv_cache_263_gb300 as pkv
from paged_kv_cache_263_gb300.workload import DeviceWorkload
from synth.workloads import small_workload
from tests.gpu_util import TOL, cache_bytes, expected_full, max_abs, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    require_gpu()


@pytest.mark.parametrize("kv_dtype,hq,hkv,qlen", [("bf16", 32, 8, 1), ("fp8", 32, 8, 1), ("bf16", 32, 8, 4),
                                                  ("bf16", 64, 8, 2), ("fp8", 16, 4, 4)])
def test_samples_of_one_prompt(kv_dtype, hq, hkv, qlen):
    prompt, gens = 1000, [37, 8, 200, 64, 9, 16]
    lens = [prompt + g for g in gens]
    wl = small_workload(1400 + qlen, lens=lens, q_lens=[qlen] * len(lens), hq=hq, hkv=hkv, kv_dtype=kv_dtype,
                        prefix_tokens=prompt, cow_block=prompt // 16)
    dw = DeviceWorkload(wl)
    tb, caches, ref = expected_full(wl)
    assert np.array_equal(dw.tables_host, tb.tables)
    assert dw.pool.stats()["cow_copies"] == len(gens) - 1
    dw.step()
    assert pkv.kv_last_device_status() == 0
    assert np.array_equal(cache_bytes(dw.k_cache), caches[0])
    assert np.array_equal(cache_bytes(dw.v_cache), caches[1])
    assert max_abs(dw.out.cpu().numpy(), ref) <= TOL[kv_dtype]
