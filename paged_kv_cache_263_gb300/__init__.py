"""GB300-native paged KV-cache attention: Python binding of libpagedkv.so.

The binding only marshals arguments: every step runs in the library (host
block manager in C++, kernels in CUDA for sm_103a).  Functions carry the
C-ABI names of ``include/pagedkv.h``; torch tensors supply device memory and
the current CUDA stream.  There is no fallback: if the library is missing or
a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "KVError", "lib", "KVPool", "kv_status_string", "reshape_and_cache",
    "paged_attention_workspace_size", "paged_attention_decode",
    "paged_attention_chunked_prefill_workspace_size", "paged_attention_chunked_prefill",
    "paged_attention_launch_count",
    "kv_last_device_status", "kv_last_device_status_flags", "KV_BF16", "KV_FP8_E4M3",
    "HEAD_DIM", "BLOCK_SIZE", "library_path", "PrefixCache", "kv_swap_out", "kv_swap_in", "kv_waste_stats",
    "kv_trace_prefill", "kv_trace_prefill_kernel_ms", "kv_selftest_bounded_wait",
]

HEAD_DIM = 128
BLOCK_SIZE = 16
KV_BF16, KV_FP8_E4M3 = 0, 1
_STATUS = {0: "ok", 1: "invalid argument", 2: "out of blocks", 3: "unsupported",
           4: "CUDA error", 5: "device data out of range"}

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libpagedkv.so")
_lib = None


class KVError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {_STATUS.get(status, status)} (status {status})")
        self.status = status


class _Stats(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("free_blocks", ctypes.c_int32),
                ("live_blocks", ctypes.c_int32), ("shared_blocks", ctypes.c_int32),
                ("cow_copies", ctypes.c_int64), ("alloc_failures", ctypes.c_int64)]


class _PrefixStats(ctypes.Structure):
    _fields_ = [("lookups", ctypes.c_int64), ("query_blocks", ctypes.c_int64),
                ("hit_blocks", ctypes.c_int64), ("inserted_blocks", ctypes.c_int64),
                ("evicted_blocks", ctypes.c_int64), ("cached_blocks", ctypes.c_int32),
                ("evictable_blocks", ctypes.c_int32)]


class _WasteStats(ctypes.Structure):
    _fields_ = [("used_tokens", ctypes.c_int64), ("contiguous_reserved_slots", ctypes.c_int64),
                ("contiguous_untouched_slots", ctypes.c_int64), ("paged_blocks", ctypes.c_int64),
                ("paged_slots", ctypes.c_int64), ("paged_waste_slots", ctypes.c_int64),
                ("contiguous_untouched_percent", ctypes.c_double), ("paged_waste_percent", ctypes.c_double)]


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(library_path):
            raise RuntimeError(f"{library_path} is not built (run __graft_entry__.build())")
        L = ctypes.CDLL(library_path)
        c = ctypes
        P, I, I64, F, SZ = c.c_void_p, c.c_int32, c.c_int64, c.c_float, c.c_size_t
        sig = {
            "kv_status_string": (c.c_char_p, [c.c_int]),
            "kv_pool_create": (c.c_int, [I, P, c.POINTER(P)]),
            "kv_pool_destroy": (None, [P]),
            "kv_block_alloc": (c.c_int, [P, I, P]),
            "kv_block_free": (c.c_int, [P, P, I]),
            "kv_block_share": (c.c_int, [P, P, I]),
            "kv_copy_on_write": (c.c_int, [P, I, c.POINTER(I), P, P, I, c.c_int, P]),
            "kv_block_refcount": (c.c_int, [P, I, c.POINTER(I)]),
            "kv_pool_stats": (c.c_int, [P, c.POINTER(_Stats)]),
            "kv_pool_fail_alloc_after": (c.c_int, [P, I]),
            "kv_waste_stats": (c.c_int, [P, I, I, c.POINTER(_WasteStats)]),
            "kv_prefix_cache_create": (c.c_int, [P, c.POINTER(P)]),
            "kv_prefix_cache_destroy": (None, [P]),
            "kv_prefix_match": (c.c_int, [P, P, I, c.c_uint64, I, P, c.POINTER(I)]),
            "kv_prefix_insert": (c.c_int, [P, P, I, c.c_uint64, P, I, c.POINTER(I)]),
            "kv_prefix_evict": (c.c_int, [P, I, P, c.POINTER(I)]),
            "kv_prefix_alloc": (c.c_int, [P, I, P]),
            "kv_prefix_stats": (c.c_int, [P, c.POINTER(_PrefixStats)]),
            "reshape_and_cache": (c.c_int, [P, P, P, P, P, I, I, I, c.c_int, P, P, P]),
            "paged_attention_workspace_size": (SZ, [I, I, I, I]),
            "paged_attention_decode": (c.c_int, [P, P, P, P, P, I, P, I, I, I, I, F, c.c_int, P, P,
                                                 I, P, SZ, P]),
            "paged_attention_chunked_prefill_workspace_size": (SZ, [I, I, I, I, I, I, I]),
            "paged_attention_launch_count": (I, [I, I, I, I, I, I, I]),
            "paged_attention_chunked_prefill": (c.c_int, [P, P, P, P, I, I, I, P, P, P, I, I, I, I,
                                                          F, c.c_int, P, P, I, P, SZ, P]),
            "paged_attention_decode_static_scratch_bytes": (SZ, []),
            "paged_attention_decode_static_scratch": (c.c_int, [P, P, P, P, P, I, P, I, I, I, I, F, c.c_int, P,
                                                                P, I, P]),
            "kv_swap_out": (c.c_int, [P, P, I, I, c.c_int, P, I, P, P, P]),
            "kv_swap_in": (c.c_int, [P, P, I, I, c.c_int, P, I, P, P, P]),
            "kv_trace_prefill": (c.c_int, [I]),
            "kv_trace_prefill_kernel_ms": (c.c_double, []),
            "kv_last_device_status": (c.c_int, [P]),
            "kv_last_device_status_flags": (c.c_uint32, []),
            "kv_selftest_bounded_wait": (c.c_int, [c.c_uint32, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(st: int, where: str):
    if st != 0:
        raise KVError(st, where)


def kv_status_string(st: int) -> str:
    return lib().kv_status_string(st).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dt(kv_dtype) -> int:
    if kv_dtype in (KV_BF16, "bf16", torch.bfloat16):
        return KV_BF16
    if kv_dtype in (KV_FP8_E4M3, "fp8", "fp8_e4m3", torch.float8_e4m3fn, torch.uint8):
        return KV_FP8_E4M3
    raise ValueError(f"unsupported kv dtype {kv_dtype}")


def _need(t, name, dtype=None, dev=True, contig=True):
    if t is None:
        raise ValueError(f"{name} is required")
    if dev and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if contig and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _cache_dtype(k_cache):
    return KV_BF16 if k_cache.dtype == torch.bfloat16 else KV_FP8_E4M3


# ------------------------------------------------------------------- pool
class KVPool:
    """Host block manager (free list, refcounts, copy-on-write)."""

    def __init__(self, num_blocks: int, initial_free_order=None):
        L = lib()
        self._p = ctypes.c_void_p()
        order = None
        if initial_free_order is not None:
            import numpy as np
            order = np.ascontiguousarray(initial_free_order, dtype=np.int32)
            if order.shape != (num_blocks,):
                raise ValueError("initial_free_order must have num_blocks entries")
        _check(L.kv_pool_create(int(num_blocks), None if order is None else order.ctypes.data_as(ctypes.c_void_p),
                                ctypes.byref(self._p)), "kv_pool_create")
        self.num_blocks = int(num_blocks)

    def close(self):
        if self._p:
            lib().kv_pool_destroy(self._p)
            self._p = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def alloc(self, n: int):
        import numpy as np
        out = np.empty(max(int(n), 0), dtype=np.int32)
        _check(lib().kv_block_alloc(self._p, int(n), out.ctypes.data_as(ctypes.c_void_p)), "kv_block_alloc")
        return out

    def free(self, ids):
        import numpy as np
        a = np.ascontiguousarray(ids, dtype=np.int32)
        _check(lib().kv_block_free(self._p, a.ctypes.data_as(ctypes.c_void_p), a.size), "kv_block_free")

    def share(self, ids):
        import numpy as np
        a = np.ascontiguousarray(ids, dtype=np.int32)
        _check(lib().kv_block_share(self._p, a.ctypes.data_as(ctypes.c_void_p), a.size), "kv_block_share")

    def copy_on_write(self, block_id: int, k_cache=None, v_cache=None, stream=None) -> int:
        """Returns the block to write into; copies K/V on the device if caches are given."""
        out = ctypes.c_int32()
        if k_cache is None:
            st = lib().kv_copy_on_write(self._p, int(block_id), ctypes.byref(out), None, None, 0, 0, None)
        else:
            _need(k_cache, "k_cache")
            _need(v_cache, "v_cache")
            st = lib().kv_copy_on_write(self._p, int(block_id), ctypes.byref(out), _ptr(k_cache),
                                        _ptr(v_cache), int(k_cache.shape[1]), _cache_dtype(k_cache),
                                        _stream(stream))
        _check(st, "kv_copy_on_write")
        return int(out.value)

    def refcount(self, block_id: int) -> int:
        out = ctypes.c_int32()
        _check(lib().kv_block_refcount(self._p, int(block_id), ctypes.byref(out)), "kv_block_refcount")
        return int(out.value)

    def stats(self) -> dict:
        s = _Stats()
        _check(lib().kv_pool_stats(self._p, ctypes.byref(s)), "kv_pool_stats")
        return {"num_blocks": s.num_blocks, "free": s.free_blocks, "live": s.live_blocks,
                "shared": s.shared_blocks, "cow_copies": s.cow_copies, "alloc_failures": s.alloc_failures}

    def fail_alloc_after(self, k: int):
        _check(lib().kv_pool_fail_alloc_after(self._p, int(k)), "kv_pool_fail_alloc_after")


def kv_waste_stats(lens, reservation_tokens: int) -> dict:
    """Contiguous-vs-paged memory waste of requests of the given lengths."""
    import numpy as np
    a = np.ascontiguousarray(lens, dtype=np.int32)
    w = _WasteStats()
    _check(lib().kv_waste_stats(a.ctypes.data_as(ctypes.c_void_p), a.size, int(reservation_tokens),
                                ctypes.byref(w)), "kv_waste_stats")
    return {f: getattr(w, f) for f, _ in _WasteStats._fields_}


class PrefixCache:
    """Block-hash prefix cache over a KVPool (kept alive by this object): exact,
    block-aligned matching from the first token under a tenant key, LRU
    eviction of leaves that only the cache holds."""

    def __init__(self, pool: KVPool):
        self.pool = pool
        self._c = ctypes.c_void_p()
        _check(lib().kv_prefix_cache_create(pool._p, ctypes.byref(self._c)), "kv_prefix_cache_create")

    def close(self):
        if self._c:
            lib().kv_prefix_cache_destroy(self._c)
            self._c = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @staticmethod
    def _tokens(tokens):
        import numpy as np
        return np.ascontiguousarray(tokens, dtype=np.int32)

    def match(self, tokens, salt: int = 0, max_blocks=None):
        """Ids of the longest cached prefix (one reference each for the caller)."""
        import numpy as np
        t = self._tokens(tokens)
        cap = t.size // BLOCK_SIZE if max_blocks is None else int(max_blocks)
        out = np.empty(max(cap, 0), dtype=np.int32)
        n = ctypes.c_int32()
        _check(lib().kv_prefix_match(self._c, t.ctypes.data_as(ctypes.c_void_p), t.size, int(salt) & (2**64 - 1),
                                     cap, out.ctypes.data_as(ctypes.c_void_p), ctypes.byref(n)), "kv_prefix_match")
        return out[:n.value]

    def insert(self, tokens, block_ids, salt: int = 0) -> int:
        import numpy as np
        t = self._tokens(tokens)
        b = np.ascontiguousarray(block_ids, dtype=np.int32)
        n = ctypes.c_int32()
        _check(lib().kv_prefix_insert(self._c, t.ctypes.data_as(ctypes.c_void_p), t.size, int(salt) & (2**64 - 1),
                                      b.ctypes.data_as(ctypes.c_void_p), b.size, ctypes.byref(n)),
               "kv_prefix_insert")
        return int(n.value)

    def evict(self, n: int):
        import numpy as np
        out = np.empty(max(int(n), 0), dtype=np.int32)
        k = ctypes.c_int32()
        _check(lib().kv_prefix_evict(self._c, int(n), out.ctypes.data_as(ctypes.c_void_p), ctypes.byref(k)),
               "kv_prefix_evict")
        return out[:k.value]

    def alloc(self, n: int):
        import numpy as np
        out = np.empty(max(int(n), 0), dtype=np.int32)
        _check(lib().kv_prefix_alloc(self._c, int(n), out.ctypes.data_as(ctypes.c_void_p)), "kv_prefix_alloc")
        return out

    def stats(self) -> dict:
        s = _PrefixStats()
        _check(lib().kv_prefix_stats(self._c, ctypes.byref(s)), "kv_prefix_stats")
        return {f: int(getattr(s, f)) for f, _ in _PrefixStats._fields_}


# ------------------------------------------------------------------ kernels
def reshape_and_cache(k, v, k_cache, v_cache, slot_mapping, k_scale=None, v_scale=None, stream=None):
    """Scatter K/V rows [T][Hkv][128] (bf16) into the paged caches at slot_mapping."""
    _need(k, "k", torch.bfloat16)
    _need(v, "v", torch.bfloat16)
    _need(k_cache, "k_cache", (torch.bfloat16, torch.uint8, torch.float8_e4m3fn))
    _need(v_cache, "v_cache", (torch.bfloat16, torch.uint8, torch.float8_e4m3fn))
    _need(slot_mapping, "slot_mapping", torch.int64)
    T, hkv, d = k.shape
    if d != HEAD_DIM or tuple(v.shape) != (T, hkv, d) or k_cache.shape[1:] != (hkv, BLOCK_SIZE, HEAD_DIM):
        raise ValueError("shape mismatch")
    dt = _cache_dtype(k_cache)
    _check(lib().reshape_and_cache(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping),
                                   T, hkv, k_cache.shape[0], dt, _ptr(k_scale), _ptr(v_scale),
                                   _stream(stream)), "reshape_and_cache")


def paged_attention_workspace_size(num_seqs, num_q_heads, max_blocks_per_seq, num_splits=0) -> int:
    return int(lib().paged_attention_workspace_size(num_seqs, num_q_heads, max_blocks_per_seq, num_splits))


def paged_attention_chunked_prefill_workspace_size(num_seqs, total_q_tokens, max_q_len, num_q_heads,
                                                   num_kv_heads, max_blocks_per_seq, num_splits=0) -> int:
    return int(lib().paged_attention_chunked_prefill_workspace_size(
        num_seqs, total_q_tokens, max_q_len, num_q_heads, num_kv_heads, max_blocks_per_seq, num_splits))


def paged_attention_launch_count(num_seqs, total_q_tokens, max_q_len, num_q_heads, num_kv_heads,
                                 max_blocks_per_seq, num_splits=0) -> int:
    return int(lib().paged_attention_launch_count(
        num_seqs, total_q_tokens, max_q_len, num_q_heads, num_kv_heads, max_blocks_per_seq, num_splits))


def _workspace(nbytes, device):
    if nbytes == 0:
        return None
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def paged_attention_decode(out, q, k_cache, v_cache, block_tables, context_lens, scale=None,
                           k_scale=None, v_scale=None, num_splits=0, workspace=None, stream=None):
    """Decode attention: out[B][Hq][128] fp32 from q[B][Hq][128] bf16 over the paged cache."""
    _need(out, "out", torch.float32)
    _need(q, "q", torch.bfloat16)
    _need(k_cache, "k_cache")
    _need(v_cache, "v_cache")
    _need(block_tables, "block_tables", torch.int32)
    _need(context_lens, "context_lens", torch.int32)
    B, hq, d = q.shape
    nb, hkv = k_cache.shape[0], k_cache.shape[1]
    mb = block_tables.shape[1]
    if scale is None:
        scale = HEAD_DIM ** -0.5
    need = paged_attention_workspace_size(B, hq, mb, num_splits)
    if workspace is None:
        workspace = _workspace(need, q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().paged_attention_decode(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                        mb, _ptr(context_lens), B, hq, hkv, nb, float(scale),
                                        _cache_dtype(k_cache), _ptr(k_scale), _ptr(v_scale), int(num_splits),
                                        _ptr(workspace), ws_bytes, _stream(stream)), "paged_attention_decode")
    return out


def paged_attention_decode_static_scratch(out, q, k_cache, v_cache, block_tables, context_lens, scale=None,
                                          k_scale=None, v_scale=None, num_splits=0, stream=None):
    """Decode for callers that cannot allocate device memory: same as
    paged_attention_decode, but the split partials live in the library's own
    fixed-size device array (see paged_attention_decode_static_scratch_bytes).
    Calls that overlap on the GPU share that array and must be serialised."""
    _need(out, "out", torch.float32)
    _need(q, "q", torch.bfloat16)
    _need(k_cache, "k_cache")
    _need(v_cache, "v_cache")
    _need(block_tables, "block_tables", torch.int32)
    _need(context_lens, "context_lens", torch.int32)
    B, hq, d = q.shape
    nb, hkv = k_cache.shape[0], k_cache.shape[1]
    if scale is None:
        scale = HEAD_DIM ** -0.5
    _check(lib().paged_attention_decode_static_scratch(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
        _ptr(context_lens), B, hq, hkv, nb, float(scale), _cache_dtype(k_cache), _ptr(k_scale), _ptr(v_scale),
        int(num_splits), _stream(stream)), "paged_attention_decode_static_scratch")
    return out


def paged_attention_decode_static_scratch_bytes() -> int:
    return int(lib().paged_attention_decode_static_scratch_bytes())


def paged_attention_chunked_prefill(out, q, cu_q_lens, context_lens, max_q_len, k_cache, v_cache,
                                    block_tables, scale=None, k_scale=None, v_scale=None, num_splits=0,
                                    workspace=None, stream=None):
    """Mixed chunked-prefill / decode attention over the paged cache."""
    _need(out, "out", torch.float32)
    _need(q, "q", torch.bfloat16)
    _need(cu_q_lens, "cu_q_lens", torch.int32)
    _need(context_lens, "context_lens", torch.int32)
    _need(block_tables, "block_tables", torch.int32)
    R, hq, d = q.shape
    B = context_lens.shape[0]
    nb, hkv = k_cache.shape[0], k_cache.shape[1]
    mb = block_tables.shape[1]
    if scale is None:
        scale = HEAD_DIM ** -0.5
    need = paged_attention_chunked_prefill_workspace_size(B, R, int(max_q_len), hq, hkv, mb, num_splits)
    if workspace is None:
        workspace = _workspace(need, q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().paged_attention_chunked_prefill(
        _ptr(out), _ptr(q), _ptr(cu_q_lens), _ptr(context_lens), B, R, int(max_q_len), _ptr(k_cache),
        _ptr(v_cache), _ptr(block_tables), mb, hq, hkv, nb, float(scale), _cache_dtype(k_cache),
        _ptr(k_scale), _ptr(v_scale), int(num_splits), _ptr(workspace), ws_bytes, _stream(stream)),
        "paged_attention_chunked_prefill")
    return out


def _swap_args(k_cache, v_cache, block_ids, host_k, host_v):
    _need(k_cache, "k_cache", (torch.bfloat16, torch.uint8, torch.float8_e4m3fn))
    _need(v_cache, "v_cache", (torch.bfloat16, torch.uint8, torch.float8_e4m3fn))
    _need(block_ids, "block_ids", torch.int32)
    n = block_ids.numel()
    for name, h in (("host_k", host_k), ("host_v", host_v)):
        _need(h, name, k_cache.dtype, dev=False)
        if h.is_cuda or not h.is_pinned():
            raise ValueError(f"{name} must be pinned host memory")
        if tuple(h.shape) != (n,) + tuple(k_cache.shape[1:]):
            raise ValueError(f"{name} must be [n][Hkv][16][128]")
    return n


def kv_swap_out(k_cache, v_cache, block_ids, host_k, host_v, stream=None):
    """Copy the listed blocks' K/V tiles to pinned host tensors [n][Hkv][16][128]."""
    n = _swap_args(k_cache, v_cache, block_ids, host_k, host_v)
    _check(lib().kv_swap_out(_ptr(k_cache), _ptr(v_cache), k_cache.shape[0], k_cache.shape[1],
                             _cache_dtype(k_cache), _ptr(block_ids), n, _ptr(host_k), _ptr(host_v),
                             _stream(stream)), "kv_swap_out")


def kv_swap_in(k_cache, v_cache, block_ids, host_k, host_v, stream=None):
    """Copy pinned host tensors [n][Hkv][16][128] into the listed (distinct) blocks."""
    n = _swap_args(k_cache, v_cache, block_ids, host_k, host_v)
    _check(lib().kv_swap_in(_ptr(k_cache), _ptr(v_cache), k_cache.shape[0], k_cache.shape[1],
                            _cache_dtype(k_cache), _ptr(block_ids), n, _ptr(host_k), _ptr(host_v),
                            _stream(stream)), "kv_swap_in")


def kv_trace_prefill(enable: bool):
    """Record CUDA events around the chunk kernel of each mixed call (tracing aid)."""
    _check(lib().kv_trace_prefill(1 if enable else 0), "kv_trace_prefill")


def kv_trace_prefill_kernel_ms() -> float:
    """Duration of the last traced chunk kernel in ms (waits for it); < 0 if none."""
    return float(lib().kv_trace_prefill_kernel_ms())


def kv_last_device_status(stream=None) -> int:
    """Synchronises the stream; returns 0 or 5 (device data out of range), clearing it."""
    st = lib().kv_last_device_status(_stream(stream))
    if st not in (0, 5):
        raise KVError(st, "kv_last_device_status")
    return st


def kv_last_device_status_flags() -> int:
    return int(lib().kv_last_device_status_flags())


def kv_selftest_bounded_wait(limit_us: int = 10000, stream=None) -> None:
    """Launches the failure-path self-test: a device wait that nothing ends gives
    up after limit_us and sets the timeout flag (8) in the status word."""
    _check(lib().kv_selftest_bounded_wait(int(limit_us), _stream(stream)), "kv_selftest_bounded_wait")
