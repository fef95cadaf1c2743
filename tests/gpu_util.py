"""Helpers shared by the GPU parity tests (no test functions here)."""
import numpy as np
import pytest
import torch

from oracle import model as omodel


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_263_gb300 import build
    build.build()


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def cache_bytes(t):
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.view(torch.uint8).numpy()


def expected_full(wl):
    tb = omodel.build_tables(wl)
    caches = omodel.build_cache(wl, tb)
    return tb, caches, omodel.expected_paged(wl, tb, caches)


TOL = {"bf16": 1e-2, "fp8": 5e-2}


def max_abs(a, b):
    return float(np.abs(np.asarray(a, dtype=np.float64) - np.asarray(b, dtype=np.float64)).max())


# On long contexts the softmax averages over so many keys that the outputs are
# small (|o| ~ 0.01 at 100K+ keys), and the stated max-abs bar alone would
# accept even an all-zero output.  Full-size checks therefore also bound the
# error relative to the largest output of the compared slice.
REL = {"bf16": 0.02, "fp8": 0.05}


def check_close(got, ref, kv_dtype, what=""):
    """max-abs error within the stated tolerance and within REL of max |ref|;
    returns (error, max |ref|)."""
    err = max_abs(got, ref)
    scale = float(np.abs(np.asarray(ref, dtype=np.float64)).max())
    assert err <= TOL[kv_dtype], (what, err)
    assert err <= REL[kv_dtype] * scale, (what, err, scale)
    return err, scale
