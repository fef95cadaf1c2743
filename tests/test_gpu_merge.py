"""The split-KV merge of the decode path (partials in the caller's workspace,
merged by a log-sum-exp kernel in fixed partition order).

A workspace needs no clearing and may be shared by calls of different shapes:
every partial a merge reads was written by the same call.  Outputs are compared
with the fp64 oracle (bf16 1e-2, fp8 5e-2); graph replays and repeated calls
must reproduce the first output bitwise."""
import numpy as np
import pytest
import torch

import paged_kv_cache_263_gb300 as pkv
from paged_kv_cache_263_gb300.workload import DeviceWorkload
from synth.workloads import small_workload
from tests.gpu_util import TOL, expected_full, max_abs, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    require_gpu()


def _ref(wl):
    _, _, ref = expected_full(wl)
    return ref


def _step(dw):
    dw.step()
    torch.cuda.synchronize()
    assert pkv.kv_last_device_status() == 0, pkv.kv_last_device_status_flags()
    return dw.out.cpu().numpy()


@pytest.mark.parametrize("fill", [0x00, 0xA5, 0xFF])
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_workspace_needs_no_clearing(fill, kv_dtype):
    wl = small_workload(501, lens=[3000, 77, 1500, 4100, 16], hq=16, hkv=4, kv_dtype=kv_dtype, num_splits=5)
    dw = DeviceWorkload(wl)
    assert dw.workspace is not None
    dw.workspace.fill_(fill)
    got = _step(dw)
    assert max_abs(got, _ref(wl)) <= TOL[kv_dtype]
    # a second call on the same workspace (the first call's partials in it) agrees bitwise
    again = _step(dw)
    assert np.array_equal(got, again)


def test_one_workspace_for_calls_of_different_shapes():
    """Calls of different batch shapes take turns on one workspace, each
    finding the other's partials where its own go."""
    wa = small_workload(502, lens=[5000, 20, 2600], hq=32, hkv=8, num_splits=6)
    wb = small_workload(503, lens=[900, 4000, 33, 2048, 7000], hq=8, hkv=2, num_splits=9)
    da, db = DeviceWorkload(wa), DeviceWorkload(wb)
    size = max(da.workspace.numel(), db.workspace.numel())
    ws = torch.full((size,), 0x5A, dtype=torch.uint8, device="cuda")
    da.workspace = db.workspace = ws
    ra, rb = _ref(wa), _ref(wb)
    first = {}
    for name, dw, ref in [("a", da, ra), ("b", db, rb), ("a", da, ra), ("b", db, rb), ("a", da, ra)]:
        got = _step(dw)
        assert max_abs(got, ref) <= TOL["bf16"], name
        if name in first:
            assert np.array_equal(got, first[name]), name
        first.setdefault(name, got)


def test_graph_replays_merge_bitwise():
    wl = small_workload(504, lens=[6000, 300, 2222, 4096], hq=32, hkv=8, num_splits=8)
    dw = DeviceWorkload(wl)
    eager = torch.from_numpy(_step(dw)).cuda()
    assert max_abs(eager.cpu().numpy(), _ref(wl)) <= TOL["bf16"]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        dw.attention()
    for _ in range(3):
        dw.out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert pkv.kv_last_device_status() == 0
        assert torch.equal(dw.out, eager)
    # an eager call between replays, on the same workspace
    dw.attention()
    dw.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(dw.out, eager)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_multi_row_merge_with_garbage_workspace(kv_dtype):
    """Short chunks (rows x G <= 8) run in the decode kernel's multi-row mode;
    their per-row partials merge the same way."""
    wl = small_workload(505, lens=[2500, 700, 4000], q_lens=[2, 1, 2], hq=16, hkv=4, kv_dtype=kv_dtype,
                        num_splits=4)
    dw = DeviceWorkload(wl)
    dw.workspace.fill_(0xC3)
    got = _step(dw)
    assert max_abs(got, _ref(wl)) <= TOL[kv_dtype]


def test_mixed_batch_decode_rows_merge():
    """Decode rows of a mixed batch (run beside the chunk kernel) merge their
    partitions too."""
    wl = small_workload(506, lens=[3000, 2100, 90, 5000], q_lens=[1, 200, 1, 1], hq=16, hkv=2, num_splits=6)
    dw = DeviceWorkload(wl)
    dw.workspace.fill_(0x77)
    got = _step(dw)
    assert max_abs(got, _ref(wl)) <= TOL["bf16"]
