"""fp64 CPU oracle for paged attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the cpu-baseline leg of
``bench.py`` import this package.  The CUDA library never calls it, and the
product path raises if its own extension is missing instead of falling back
here.

The numerical core is ``oracle.c`` (plain C, fp64, OpenMP over independent
sequences/heads); ``allocator.py`` models the block manager; ``model.py``
replays a synthetic workload through both to produce expected block tables,
cache bytes and attention outputs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_SRC = os.path.join(_HERE, "oracle.c")
_lock = threading.Lock()
_lib = None

BF16, FP8 = 0, 1


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, no fast-math, no FMA contraction)."""
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
           "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_SO)
            c = ctypes
            P = c.c_void_p
            L.oracle_bf16_to_f64.restype = c.c_double
            L.oracle_bf16_to_f64.argtypes = [c.c_uint16]
            L.oracle_e4m3_to_f64.restype = c.c_double
            L.oracle_e4m3_to_f64.argtypes = [c.c_uint8]
            L.oracle_e4m3_from_f32.restype = c.c_uint8
            L.oracle_e4m3_from_f32.argtypes = [c.c_float]
            L.oracle_e4m3_encode_array.restype = None
            L.oracle_e4m3_encode_array.argtypes = [P, P, c.c_int64]
            L.oracle_reshape_and_cache.restype = c.c_int
            L.oracle_reshape_and_cache.argtypes = [P, P, P, P, P, c.c_int, c.c_int, c.c_int, c.c_int,
                                                   c.c_int64, c.c_int, P, P]
            L.oracle_contiguous_attention.restype = c.c_int
            L.oracle_contiguous_attention.argtypes = [P, P, P, P, c.c_int, c.c_int64, c.c_int, c.c_int,
                                                      c.c_int, c.c_double, c.c_int]
            L.oracle_paged_attention.restype = c.c_int
            L.oracle_paged_attention.argtypes = [P, P, P, P, c.c_int, P, P, P, c.c_int, P, P, c.c_int,
                                                 c.c_int, c.c_int, c.c_int, c.c_int, c.c_int64,
                                                 c.c_double, c.c_int]
            L.oracle_max_threads.restype = c.c_int
            L.oracle_max_threads.argtypes = []
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    return int(lib().oracle_max_threads())


# ------------------------------------------------------------------ formats
def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact fp64 values."""
    u = (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16)
    return u.view(np.float32).astype(np.float64)


def e4m3_decode(codes) -> np.ndarray:
    L = lib()
    codes = np.asarray(codes, dtype=np.uint8)
    table = np.array([L.oracle_e4m3_to_f64(i) for i in range(256)], dtype=np.float64)
    return table[codes]


def e4m3_encode(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().oracle_e4m3_encode_array(_p(x), _p(out), x.size)
    return out


# ---------------------------------------------------------------- the path
def reshape_and_cache(k_bits, v_bits, k_cache, v_cache, slot_mapping, dtype=BF16,
                      k_scale=None, v_scale=None):
    """In-place scatter of K/V rows [T][Hkv][D] (bf16 bits) into the caches."""
    k_bits = np.ascontiguousarray(k_bits, dtype=np.uint16)
    v_bits = np.ascontiguousarray(v_bits, dtype=np.uint16)
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    T, Hkv, D = k_bits.shape
    nb, hk, bs, dd = k_cache.shape
    assert hk == Hkv and dd == D and k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    ks = None if k_scale is None else np.ascontiguousarray(k_scale, dtype=np.float32)
    vs = None if v_scale is None else np.ascontiguousarray(v_scale, dtype=np.float32)
    rc = lib().oracle_reshape_and_cache(_p(k_bits), _p(v_bits), _p(k_cache), _p(v_cache), _p(slots),
                                        T, Hkv, D, bs, nb, dtype, _p(ks), _p(vs))
    if rc != 0:
        raise ValueError("slot outside the pool")


def paged_attention(q_bits, k_cache, v_cache, block_tables, context_lens, cu_q_lens=None,
                    num_q_heads=None, dtype=BF16, k_scale=None, v_scale=None, scale=None,
                    nthreads=0) -> np.ndarray:
    """fp64 [R][Hq][D] outputs of paged attention (see oracle.c)."""
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    R, Hq, D = q_bits.shape
    nb, Hkv, bs, dd = k_cache.shape
    assert dd == D
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    cu = None if cu_q_lens is None else np.ascontiguousarray(cu_q_lens, dtype=np.int32)
    B = len(cl)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    ks = None if k_scale is None else np.ascontiguousarray(k_scale, dtype=np.float32)
    vs = None if v_scale is None else np.ascontiguousarray(v_scale, dtype=np.float32)
    out = np.zeros((R, Hq, D), dtype=np.float64)
    rc = lib().oracle_paged_attention(_p(out), _p(q_bits), _p(np.ascontiguousarray(k_cache)),
                                      _p(np.ascontiguousarray(v_cache)), dtype, _p(ks), _p(vs),
                                      _p(bt), bt.shape[1], _p(cl), _p(cu), B, Hq, Hkv, D, bs, nb,
                                      float(scale), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_paged_attention failed ({rc})")
    return out


def contiguous_attention(q, k, v, scale=None, nthreads=0) -> np.ndarray:
    """fp64 textbook attention of one sequence: q [n][Hq][D], k/v [L][Hkv][D]."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    n, Hq, D = q.shape
    L, Hkv, _ = k.shape
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    out = np.zeros((n, Hq, D), dtype=np.float64)
    rc = lib().oracle_contiguous_attention(_p(out), _p(q), _p(k), _p(v), n, L, Hq, Hkv, D,
                                           float(scale), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_contiguous_attention failed")
    return out
