"""Full-size workloads on the GPU, checked on sampled outputs that the oracle
computes one by one (contiguous fp64 attention on the generator's values),
plus bit-exact block tables and sampled cache bytes."""
import numpy as np
import pytest
import torch

import oracle
from oracle import model as omodel
from paged_kv_cache_263_gb300.workload import DeviceWorkload
import paged_kv_cache_263_gb300 as pkv
from synth.workloads import DISTINCT_FP8_FACTORS, make_workload
from tests.gpu_util import TOL, cache_bytes, check_close, max_abs, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    require_gpu()


def _check_cache_samples(wl, dw, tb, n=2000, seed=0):
    rng = np.random.default_rng(seed)
    B = wl.num_seqs
    kc = dw.k_cache
    vc = dw.v_cache
    ss = rng.integers(0, B, size=n)
    ts = np.array([rng.integers(0, int(wl.context_lens[s])) for s in ss])
    blk = tb.tables[ss, ts // 16]
    off = ts % 16
    keys = np.array([wl.token_keys(s, t, t + 1)[0] for s, t in zip(ss, ts)])
    k = wl.kv_values("k", keys)
    v = wl.kv_values("v", keys)
    idx_b = torch.from_numpy(blk.astype(np.int64)).cuda()
    idx_o = torch.from_numpy(off.astype(np.int64)).cuda()
    got_k = cache_bytes(kc[idx_b, :, idx_o])
    got_v = cache_bytes(vc[idx_b, :, idx_o])
    if wl.kv_dtype == "fp8":
        ks, vs = wl.fp8_scales()
        ref_k = oracle.e4m3_encode(k.float().numpy() / ks[None, :, None])
        ref_v = oracle.e4m3_encode(v.float().numpy() / vs[None, :, None])
    else:
        ref_k = k.contiguous().view(torch.int16).numpy().view(np.uint16)
        ref_v = v.contiguous().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got_k, ref_k)
    assert np.array_equal(got_v, ref_v)


def _check(name, sample_seqs, nthreads=0, fp8_scale_factors=None):
    wl = make_workload(name, fp8_scale_factors=fp8_scale_factors)
    tb = omodel.build_tables(wl)
    dw = DeviceWorkload(wl)
    assert np.array_equal(dw.tables_host, tb.tables)
    dw.step()
    assert pkv.kv_last_device_status() == 0
    _check_cache_samples(wl, dw, tb)
    out = dw.out.cpu().numpy()
    cu = wl.cu_q_lens
    worst = 0.0
    for s in sample_seqs:
        ref = omodel.expected_rows(wl, s, nthreads=nthreads)
        got = out[cu[s]:cu[s + 1]]
        err, _ = check_close(got, ref, wl.kv_dtype, (name, s))
        worst = max(worst, err)
    return dw, worst


def test_llama8b_decode():
    wl = make_workload("llama8b")
    order = np.argsort(wl.context_lens)
    _check("llama8b", [int(order[0]), int(order[-1]), 7, 31, 63])


def test_llama70b_shared_prefix_decode():
    wl = make_workload("llama70b_prefix")
    order = np.argsort(wl.context_lens)
    dw, _ = _check("llama70b_prefix", [int(order[0]), int(order[-1]), 0, 127])
    # the copy-on-write fork left every sharer pointing at the same 124 prefix blocks
    t = dw.tables_host
    assert (t[:, :124] == t[0, :124]).all()
    assert len(set(t[:, 124].tolist())) == 128
    assert dw.pool.stats()["cow_copies"] == 127


def test_split_kv_fp8_long_context():
    _, _ = _check("split_fp8", [0, 5])


def test_split_kv_fp8_long_context_distinct_per_head_scales():
    """The full-size split-KV fp8 batch with K and V scales that differ by head
    and by tensor (up to 8x): sampled sequences against the oracle, and the
    oracle with the K and V scales swapped is far from the GPU output."""
    dw, _ = _check("split_fp8", [2, 7], fp8_scale_factors=DISTINCT_FP8_FACTORS)
    wl = dw.wl
    ks, vs = wl.fp8_scales()
    assert (ks != vs).all() and len(set(ks.tolist())) == len(set(vs.tolist())) == 8
    got = dw.out.cpu().numpy()
    assert max_abs(got[2:3], omodel.expected_rows(wl, 2, dequant=(vs, ks))) > 4 * TOL["fp8"]
