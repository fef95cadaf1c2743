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
