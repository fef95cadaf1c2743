"""Failure detection on the GPU without a fault: a device wait that nothing
ends (an mbarrier phase no thread completes) gives up after its limit, sets the
timeout flag in the status word, and leaves the context usable -- the next
status read is clean and attention still matches the oracle."""
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


def test_bounded_wait_gives_up_and_reports():
    torch.cuda.synchronize()
    pkv.kv_last_device_status()                      # drain whatever an earlier test left
    pkv.kv_selftest_bounded_wait(10_000)            # 10 ms
    assert pkv.kv_last_device_status() == 5          # KV_ERR_DEVICE_BOUNDS
    assert pkv.kv_last_device_status_flags() & 8     # the timeout flag
    assert pkv.kv_last_device_status() == 0          # read and cleared
    # the context still computes
    wl = small_workload(601, lens=[700, 33, 2100], hq=8, hkv=2, num_splits=3)
    dw = DeviceWorkload(wl)
    dw.step()
    assert pkv.kv_last_device_status() == 0
    _, _, ref = expected_full(wl)
    assert max_abs(dw.out.cpu().numpy(), ref) <= TOL["bf16"]
