"""fp8-e4m3 cache with per-KV-head scales that differ between K and V and from
head to head ("Waste, and three ways to reclaim it", "Quantising the cache";
"M.65 Inference serving", quantisation (b), (d)): every fp8 attention path --
the decode kernel, its multi-row mode for short chunks, and the tensor-core
chunk kernel -- must dequantise K with k_scale[g] and V with v_scale[g] of the
query head's own KV head g.

Besides parity with the fp64 oracle, each case shows that it would catch the
plausible mistakes: the oracle run with K and V scales swapped, with head 0's
scales for every head, or with the heads' scales reversed, lands far outside
the tolerance of the GPU output.  The mistakes are planted in the oracle's
inputs on the CPU; the GPU runs the library as built.

It also checks the range of the query that the fp8 paths accept: they round Q
from bf16 to f16 once, which is exact for 2^-14 <= |q| < 65,520, loses low bits
of smaller components (f16 subnormals) and overflows at |q| >= 65,520."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_263_gb300 as pkv
from oracle import model as omodel
from paged_kv_cache_263_gb300.workload import DeviceWorkload
from synth.workloads import DISTINCT_FP8_FACTORS, small_workload
from tests.gpu_util import TOL, bits, cache_bytes, max_abs, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    require_gpu()


def _oracle(wl, tb, caches, ks, vs, q_bits=None):
    q = bits(wl.q_values()) if q_bits is None else q_bits
    cu = None if wl.is_decode else wl.cu_q_lens
    return oracle.paged_attention(q, caches[0], caches[1], tb.tables, wl.context_lens, cu, dtype=oracle.FP8,
                                  k_scale=ks, v_scale=vs, scale=wl.scale)


def _check(wl, q_scale=None, plant=True):
    """GPU output vs the oracle with the right scales, and (``plant``) far from
    it with planted scale mistakes.  Returns the error against the right oracle."""
    tb = omodel.build_tables(wl)
    dw = DeviceWorkload(wl)
    caches = omodel.build_cache(wl, tb)
    assert np.array_equal(dw.tables_host, tb.tables)
    q_bits = None
    if q_scale is not None:
        q = (wl.q_values().float() * q_scale).to(torch.bfloat16)
        dw.q.copy_(q.to(dw.q.device))
        q_bits = bits(q)
    dw.step()                                   # writes the step's new tokens, then attends
    assert pkv.kv_last_device_status() == 0
    # the cache the kernels read holds the oracle's bytes (per-head scales at the write)
    assert np.array_equal(cache_bytes(dw.k_cache), caches[0])
    assert np.array_equal(cache_bytes(dw.v_cache), caches[1])
    got = dw.out.cpu().numpy().astype(np.float64)
    ks, vs = wl.fp8_scales()
    # K and V scales differ head by head, and the heads' scales differ from each other
    assert (ks != vs).all() and len(set(ks.tolist())) == len(set(vs.tolist())) == wl.num_kv_heads
    err = max_abs(got, _oracle(wl, tb, caches, ks, vs, q_bits))
    assert err <= TOL["fp8"], err
    if not plant:
        return err
    mistakes = {
        "k and v swapped": (vs, ks),
        "head 0 for all": (np.full_like(ks, ks[0]), np.full_like(vs, vs[0])),
        "heads reversed": (ks[::-1].copy(), vs[::-1].copy()),
    }
    for name, (mk, mv) in mistakes.items():
        wrong = max_abs(got, _oracle(wl, tb, caches, mk, mv, q_bits))
        assert wrong > 4 * TOL["fp8"], (name, wrong)
    return err


LENS = [1, 2, 15, 16, 17, 40, 130, 700, 2100]


@pytest.mark.parametrize("hq,hkv,splits", [(8, 2, 0), (16, 2, 3), (64, 8, 0), (64, 8, 5), (32, 8, 1)])
def test_decode_uses_each_heads_own_k_and_v_scale(hq, hkv, splits):
    wl = small_workload(1100 + hq + splits, lens=LENS, hq=hq, hkv=hkv, kv_dtype="fp8", num_splits=splits,
                        fp8_scale_factors=DISTINCT_FP8_FACTORS)
    _check(wl)


@pytest.mark.parametrize("hq,hkv,n", [(8, 2, 2), (32, 8, 2), (16, 8, 4), (8, 8, 8), (8, 2, 4), (16, 8, 8)])
def test_multi_row_mode_uses_each_heads_own_k_and_v_scale(hq, hkv, n):
    # max_q_len * G <= 8: the short chunks run in the decode kernel's multi-row
    # mode; 16 columns (the last two cases) take the tensor-core kernel
    lens = [n, n + 1, 30, 300, 1500]
    wl = small_workload(1200 + hq + n, lens=lens, q_lens=[n] * len(lens), hq=hq, hkv=hkv, kv_dtype="fp8",
                        fp8_scale_factors=DISTINCT_FP8_FACTORS)
    _check(wl)


@pytest.mark.parametrize("hq,hkv,q_lens", [(64, 8, [130, 1, 1, 3]), (32, 8, [200, 1, 64, 1]),
                                           (8, 2, [300, 1, 1, 1])])
def test_tensor_core_chunk_uses_each_heads_own_k_and_v_scale(hq, hkv, q_lens):
    lens = [2600, 17, 900, 65]
    wl = small_workload(1300 + hq, lens=lens, q_lens=q_lens, hq=hq, hkv=hkv, kv_dtype="fp8",
                        fp8_scale_factors=DISTINCT_FP8_FACTORS)
    _check(wl)


@pytest.mark.parametrize("q_scale", [1000.0, 2.0 ** -12])
@pytest.mark.parametrize("q_lens", [[1, 1, 1], [3, 3, 3], [130, 1, 2]], ids=["decode", "multirow", "chunk"])
def test_fp8_paths_accept_large_and_small_queries(q_scale, q_lens):
    """Queries of N(0,1)-shaped values x 1000 (|q| up to ~3,500: the rounding to
    f16 is exact, scores in the thousands make the softmax nearly one-hot) and
    x 2^-12 (most components in f16's subnormal range, where the rounding drops
    low bits; every score is near 0): the fp8 paths keep parity with the oracle,
    which uses the bf16 query exactly.  |q| >= 65,520 would overflow f16; the
    header states that limit."""
    lens = [700, 150, 2000]
    hq, hkv = (8, 2) if q_lens[0] <= 3 else (32, 8)
    wl = small_workload(1400, lens=lens, q_lens=q_lens, hq=hq, hkv=hkv, kv_dtype="fp8",
                        fp8_scale_factors=DISTINCT_FP8_FACTORS)
    # (a tiny q makes every score ~0: the output is the mean of V, which the
    # planted mistakes move too little to be a useful check here)
    _check(wl, q_scale=q_scale, plant=q_scale > 1)
