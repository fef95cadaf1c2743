"""Paging does not change the result ("Waste, and three ways to reclaim it",
section "PagedAttention": the kernel reads the same values through the table,
wherever the blocks sit).  At the full sizes of every workload, in the launch
configuration the benchmark times -- the partition plans chosen for those sizes,
the multi-row mode, the tensor-core chunk kernel and the decode rows that run
beside it --, the same batch is placed by three different seeded permutations of
the physical pool and the whole output must be bitwise identical.  The
comparison is made on the device; no oracle is involved."""
import numpy as np
import pytest
import torch

import paged_kv_cache_263_gb300 as pkv
from paged_kv_cache_263_gb300.workload import DeviceWorkload
from synth.workloads import make_workload
from tests.gpu_util import require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    require_gpu()


WORKLOADS = ["llama8b", "llama70b_prefix", "mixed_prefill", "mixed_prefill_fp8", "split_fp8",
             "spec_verify", "spec_verify8"]


@pytest.mark.parametrize("name", WORKLOADS)
def test_full_size_output_is_bitwise_identical_under_three_placements(name):
    outs, scales = [], None
    for perm_seed in (11, 12, 13):
        wl = make_workload(name)
        wl.free_order = np.random.default_rng(perm_seed).permutation(wl.num_blocks).astype(np.int32)
        if scales is not None:
            wl._fp8_scales = scales           # values (and so scales) do not depend on placement
        dw = DeviceWorkload(wl)
        if wl.kv_dtype == "fp8":
            scales = wl._fp8_scales
        dw.step()
        assert pkv.kv_last_device_status() == 0
        out = dw.out.clone()
        assert torch.isfinite(out).all()
        outs.append(out)
        del dw
        torch.cuda.empty_cache()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
