"""The five synthetic paged-attention workloads, as plain data.

Every workload is seeded (seed = 2630 + its number) and describes only the
*inputs*: sequence lengths, query-chunk lengths, the order in which physical
blocks are handed out by the pool, the shared prefix, the copy-on-write fork,
and the counter-based value streams for Q, K and V.  Building block tables,
writing the cache and computing attention are left to the two sides (the CUDA
library and the oracle), each with its own code.

Recipes (the shapes follow Llama-3 layers; "1K" = 1,024 tokens):

1. ``tiny``      4 sequences of 300/2,000/600/4,400 tokens; Hq 8, Hkv 2; pool of
                 512 blocks handed out in a seeded random order; bf16.
2. ``llama8b``   64 sequences, length uniform in [512, 4096]; Hq 32, Hkv 8;
                 pool of 65,536 blocks in random order; bf16.
3. ``llama70b_prefix``  128 sequences sharing one 2,000-token prefix (125 blocks,
                 ref-counted), then a private tail of floor(exp(U[ln 1K, ln 32K]))
                 tokens; Hq 64, Hkv 8; each sequence forks logical block 124 with
                 copy-on-write before its tail is written; bf16.
4. ``mixed_prefill``  one 1,024-token query chunk over 100,000 cached tokens
                 (context 101,024) plus 255 decode sequences of length uniform in
                 [1K, 8K]; Hq 64, Hkv 8; bf16.
5. ``split_fp8`` 8 sequences of 131,072 tokens; Hq 64, Hkv 8; fp8-e4m3 cache with
                 per-head scales; 16 split-KV partitions.

Further shapes: ``spec_verify`` (64 sequences of the ``llama8b`` recipe, each
verifying a 4-token draft: 4 causal query rows per sequence) and
``spec_verify8`` (32 sequences, lengths uniform in [1K, 8K], Hq 64, Hkv 8,
8-token drafts) -- speculative decoding's verification pass ("M.65 Inference
serving", speculative decoding: a draft of N = 4-8 tokens verified in one
forward pass); ``mixed_prefill_small`` (the mixed batch scaled down for
profiling); ``prefill_chunk`` (the mixed batch's chunk without its decode
rows: the tensor-core kernel alone); ``prefill_chunk_small`` (the chunk of
``mixed_prefill_small`` alone, for full profiler captures of that kernel on
every SM).

fp8 workloads carry per-KV-head scales for K and for V (``fp8_scales``):
amax / 448 over every value of that head and tensor in the workload.

For every sequence the step's "new" tokens (the last ``q_len`` positions) are
the ones appended by the cache write in the step; all earlier positions are
written while the workload is set up.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

from . import normal_bf16, stream_key

__all__ = ["Workload", "make_workload", "WORKLOADS", "EXTRA_WORKLOADS", "small_workload",
           "DISTINCT_FP8_FACTORS", "E4M3_MAX"]

Q_STREAM, K_STREAM, V_STREAM = 0, 1, 2

E4M3_MAX = np.float32(448.0)          # largest finite e4m3 magnitude

# Per-(tensor, KV head) multipliers of the fp8 scales for parity tests of the
# scale path: K and V scales then differ from each other and from head to head
# by up to 8x, so a kernel that swapped them, or read one head's scale for
# another, would be far outside the tolerance.  Factors below 1 make the
# largest values saturate at 448, which is part of what the tests exercise.
DISTINCT_FP8_FACTORS = (
    np.array([1.0, 2.5, 0.5, 4.0, 0.75, 3.0, 1.5, 0.625], dtype=np.float32),   # K, head 0..7
    np.array([3.0, 0.5, 2.0, 0.625, 4.0, 1.0, 0.75, 2.5], dtype=np.float32),   # V, head 0..7
)


@dataclass
class Workload:
    name: str
    seed: int
    num_q_heads: int
    num_kv_heads: int
    num_blocks: int
    kv_dtype: str                    # "bf16" or "fp8"
    context_lens: np.ndarray         # int32 [B]; includes the step's new tokens
    q_lens: np.ndarray               # int32 [B]; 1 for decode rows
    free_order: np.ndarray           # int32 [num_blocks]; first entry is handed out first
    prefix_tokens: int = 0           # tokens of one prefix shared by every sequence
    cow_block: int = -1              # logical block forked by copy-on-write (-1: none)
    num_splits: int = 0              # split-KV partitions per sequence (0: library picks)
    head_dim: int = 128
    block_size: int = 16
    description: str = ""
    fp8_scale_factors: tuple = None  # (K [Hkv], V [Hkv]) fp32 multipliers of the amax scales
    _tail_base: np.ndarray = field(default=None, repr=False)
    _fp8_scales: tuple = field(default=None, repr=False)

    def __post_init__(self):
        self.context_lens = np.asarray(self.context_lens, dtype=np.int32)
        self.q_lens = np.asarray(self.q_lens, dtype=np.int32)
        self.free_order = np.asarray(self.free_order, dtype=np.int32)
        tails = (self.context_lens.astype(np.int64) - self.prefix_tokens)
        base = np.zeros(len(tails), dtype=np.int64)
        if len(tails) > 1:
            base[1:] = np.cumsum(tails)[:-1]
        self._tail_base = base + self.prefix_tokens

    # ------------------------------------------------------------------ sizes
    @property
    def num_seqs(self) -> int:
        return int(len(self.context_lens))

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def total_q(self) -> int:
        return int(self.q_lens.sum())

    @property
    def cu_q_lens(self) -> np.ndarray:
        cu = np.zeros(self.num_seqs + 1, dtype=np.int32)
        cu[1:] = np.cumsum(self.q_lens)
        return cu

    @property
    def max_blocks_per_seq(self) -> int:
        return int(-(-int(self.context_lens.max()) // self.block_size))

    @property
    def is_decode(self) -> bool:
        return bool((self.q_lens == 1).all())

    @property
    def kv_elem_bytes(self) -> int:
        return 1 if self.kv_dtype == "fp8" else 2

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    # ------------------------------------------------------------ value keys
    def token_keys(self, s: int, t0: int, t1: int) -> np.ndarray:
        """Value-stream keys of tokens t0..t1-1 of sequence s (prefix tokens are
        the same logical tokens in every sequence)."""
        t = np.arange(t0, t1, dtype=np.int64)
        key = self._tail_base[s] + (t - self.prefix_tokens)
        if self.prefix_tokens:
            key = np.where(t < self.prefix_tokens, t, key)
        return key

    def kv_values(self, which: str, keys, device="cpu") -> torch.Tensor:
        """bf16 [len(keys)][Hkv][D] K or V rows for the given token keys."""
        sid = K_STREAM if which == "k" else V_STREAM
        keys = torch.as_tensor(np.asarray(keys, dtype=np.int64), device=device)
        hd = self.num_kv_heads * self.head_dim
        ctr = keys[:, None] * hd + torch.arange(hd, device=device, dtype=torch.int64)[None, :]
        out = normal_bf16(stream_key(self.seed, sid), ctr)
        return out.view(len(keys), self.num_kv_heads, self.head_dim)

    def seq_kv(self, which: str, s: int, t0: int = 0, t1: int | None = None, device="cpu"):
        if t1 is None:
            t1 = int(self.context_lens[s])
        return self.kv_values(which, self.token_keys(s, t0, t1), device)

    def q_values(self, rows=None, device="cpu") -> torch.Tensor:
        """bf16 [rows][Hq][D] query rows (global row index over all sequences)."""
        if rows is None:
            rows = np.arange(self.total_q, dtype=np.int64)
        rows = torch.as_tensor(np.asarray(rows, dtype=np.int64), device=device)
        hd = self.num_q_heads * self.head_dim
        ctr = rows[:, None] * hd + torch.arange(hd, device=device, dtype=torch.int64)[None, :]
        out = normal_bf16(stream_key(self.seed, Q_STREAM), ctr)
        return out.view(len(rows), self.num_q_heads, self.head_dim)

    @property
    def unique_tokens(self) -> int:
        """Distinct logical tokens of the workload: the shared prefix once plus
        every sequence's own tokens.  Their value-stream keys are exactly
        0 .. unique_tokens - 1 (see token_keys)."""
        return int(self.prefix_tokens + (self.context_lens.astype(np.int64) - self.prefix_tokens).sum())

    def kv_amax(self, device="cpu", chunk_tokens=1 << 15):
        """Per-KV-head max |x| of the K and of the V values of every token of the
        workload (bf16 values, so exact in fp32): two fp32 arrays [Hkv].  A max
        is exact, so the result does not depend on the device that scans."""
        ka = torch.zeros(self.num_kv_heads, dtype=torch.float32, device=device)
        va = torch.zeros_like(ka)
        n = self.unique_tokens
        for a in range(0, n, chunk_tokens):
            keys = np.arange(a, min(n, a + chunk_tokens), dtype=np.int64)
            for which, acc in (("k", ka), ("v", va)):
                x = self.kv_values(which, keys, device).float().abs()
                torch.maximum(acc, x.amax(dim=(0, 2)), out=acc)
        return ka.cpu().numpy(), va.cpu().numpy()

    def fp8_scales(self, device=None):
        """Per-KV-head fp32 scales of K and of V for the fp8-e4m3 cache.

        The reading taken for the scale (the pages leave it open): one scale per
        KV head and per tensor, s = amax / 448 over all of that head's values
        in the workload (IEEE fp32 division), so the largest value maps to the
        largest finite e4m3 magnitude.  With ``fp8_scale_factors`` set, each
        scale is then multiplied (fp32) by its factor.  Computed once and kept;
        the scan runs on ``device`` (default: the GPU if torch has one, else
        the CPU -- the max is exact, so both give the same bits)."""
        if self._fp8_scales is None:
            if device is None:
                device = "cuda" if torch.cuda.is_available() else "cpu"
            ka, va = self.kv_amax(device)
            ks = (ka.astype(np.float32) / E4M3_MAX).astype(np.float32)
            vs = (va.astype(np.float32) / E4M3_MAX).astype(np.float32)
            if self.fp8_scale_factors is not None:
                kf, vf = self.fp8_scale_factors
                ks = (ks * np.resize(np.asarray(kf, np.float32), self.num_kv_heads)).astype(np.float32)
                vs = (vs * np.resize(np.asarray(vf, np.float32), self.num_kv_heads)).astype(np.float32)
            self._fp8_scales = (ks, vs)
        ks, vs = self._fp8_scales
        return ks.copy(), vs.copy()

    # ------------------------------------------------------------ bytes
    def kv_bytes_per_token(self) -> int:
        return 2 * self.num_kv_heads * self.head_dim * self.kv_elem_bytes

    def summary(self) -> dict:
        return {
            "workload": self.name, "num_seqs": self.num_seqs, "num_q_heads": self.num_q_heads,
            "num_kv_heads": self.num_kv_heads, "head_dim": self.head_dim,
            "block_size": self.block_size, "kv_dtype": self.kv_dtype,
            "num_blocks": self.num_blocks, "total_context_tokens": int(self.context_lens.sum()),
            "total_q_tokens": self.total_q, "prefix_tokens": self.prefix_tokens,
            "num_splits": self.num_splits,
        }


def _blocks(n, bs=16):
    return -(-int(n) // bs)


def _pool_to_fit(lens, prefix, cow, bs=16, slack=1.02):
    need = 0
    pb = _blocks(prefix, bs) if prefix else 0
    for L in lens:
        need += _blocks(L, bs) - pb
    need += pb
    if cow >= 0:
        need += len(lens)
    return int(math.ceil(need * slack / 1024.0) * 1024)


def make_workload(name: str, fp8_scale_factors=None) -> Workload:
    """The named workload; ``fp8_scale_factors`` (K, V multipliers per KV head)
    changes the fp8 scales of an fp8 workload (see Workload.fp8_scales)."""
    wl = _make(name)
    wl.fp8_scale_factors = fp8_scale_factors
    return wl


def _make(name: str) -> Workload:
    if name in ("tiny", "cfg1", "1"):
        seed = 2631
        rng = np.random.Generator(np.random.PCG64(seed))
        lens = np.array([300, 2000, 600, 4400], dtype=np.int32)
        pool = 512
        return Workload("tiny", seed, 8, 2, pool, "bf16", lens, np.ones(4, np.int32),
                        rng.permutation(pool), description="tiny paged decode, GQA 4")
    if name in ("llama8b", "cfg2", "2"):
        seed = 2632
        rng = np.random.Generator(np.random.PCG64(seed))
        lens = rng.integers(512, 4096, size=64, endpoint=True).astype(np.int32)
        pool = 65536
        return Workload("llama8b", seed, 32, 8, pool, "bf16", lens, np.ones(64, np.int32),
                        rng.permutation(pool), description="Llama-3-8B layer-shape decode, batch 64")
    if name in ("llama70b_prefix", "cfg3", "3"):
        seed = 2633
        rng = np.random.Generator(np.random.PCG64(seed))
        u = rng.uniform(math.log(1024), math.log(32768), size=128)
        tails = np.floor(np.exp(u)).astype(np.int64)
        lens = (2000 + tails).astype(np.int32)
        pool = _pool_to_fit(lens, 2000, 124)
        return Workload("llama70b_prefix", seed, 64, 8, pool, "bf16", lens,
                        np.ones(128, np.int32), rng.permutation(pool), prefix_tokens=2000,
                        cow_block=124,
                        description="Llama-3-70B layer-shape decode, batch 128, shared 2,000-token prefix")
    if name in ("mixed_prefill", "cfg4", "4"):
        seed = 2634
        rng = np.random.Generator(np.random.PCG64(seed))
        dec = rng.integers(1024, 8192, size=255, endpoint=True).astype(np.int32)
        lens = np.concatenate([[101024], dec]).astype(np.int32)
        qlens = np.concatenate([[1024], np.ones(255, np.int64)]).astype(np.int32)
        pool = _pool_to_fit(lens, 0, -1)
        return Workload("mixed_prefill", seed, 64, 8, pool, "bf16", lens, qlens,
                        rng.permutation(pool),
                        description="chunked-prefill mix: 1,024-token chunk over 100,000 cached tokens + 255 decodes")
    if name == "mixed_prefill_small":
        # the mixed batch scaled down for profiling: one 1,024-token chunk over
        # 40,000 cached tokens plus 63 decodes (KV ~0.3 GB, still above L2)
        seed = 2644
        rng = np.random.Generator(np.random.PCG64(seed))
        dec = rng.integers(1024, 8192, size=63, endpoint=True).astype(np.int32)
        lens = np.concatenate([[41024], dec]).astype(np.int32)
        qlens = np.concatenate([[1024], np.ones(63, np.int64)]).astype(np.int32)
        pool = _pool_to_fit(lens, 0, -1)
        return Workload("mixed_prefill_small", seed, 64, 8, pool, "bf16", lens, qlens,
                        rng.permutation(pool),
                        description="chunked-prefill mix for profiling: 1,024-token chunk over 40,000 cached tokens + 63 decodes")
    if name in ("split_fp8", "cfg5", "5"):
        seed = 2635
        rng = np.random.Generator(np.random.PCG64(seed))
        lens = np.full(8, 131072, dtype=np.int32)
        pool = 65536
        return Workload("split_fp8", seed, 64, 8, pool, "fp8", lens, np.ones(8, np.int32),
                        rng.permutation(pool), num_splits=16,
                        description="long-context split-KV decode, fp8-e4m3 cache, 16 partitions")
    if name == "mixed_prefill_small_fp8":
        wl = _make("mixed_prefill_small")
        wl.name, wl.kv_dtype, wl.seed = "mixed_prefill_small_fp8", "fp8", 2645
        wl.description = "the profiling mix over an fp8-e4m3 cache"
        return wl
    if name == "mixed_prefill_fp8":
        # the chunked-prefill mix with an fp8-e4m3 cache
        wl = _make("mixed_prefill")
        wl.name, wl.kv_dtype, wl.seed = "mixed_prefill_fp8", "fp8", 2639
        wl.description = "chunked-prefill mix over an fp8-e4m3 cache"
        return wl
    if name == "spec_verify":
        # speculative-decoding verification at the Llama-3-8B layer shape: every
        # sequence checks a 4-token draft in one pass (4 causal query rows)
        seed = 2637
        rng = np.random.Generator(np.random.PCG64(seed))
        lens = rng.integers(512, 4096, size=64, endpoint=True).astype(np.int32)
        pool = 65536
        return Workload("spec_verify", seed, 32, 8, pool, "bf16", lens, np.full(64, 4, np.int32),
                        rng.permutation(pool),
                        description="speculative verify: 64 sequences x 4 draft tokens, Llama-3-8B layer shape")
    if name == "spec_verify8":
        # the same at the Llama-3-70B layer shape with an 8-token draft
        seed = 2638
        rng = np.random.Generator(np.random.PCG64(seed))
        lens = rng.integers(1024, 8192, size=32, endpoint=True).astype(np.int32)
        pool = _pool_to_fit(lens, 0, -1)
        return Workload("spec_verify8", seed, 64, 8, pool, "bf16", lens, np.full(32, 8, np.int32),
                        rng.permutation(pool),
                        description="speculative verify: 32 sequences x 8 draft tokens, Llama-3-70B layer shape")
    if name == "prefill_chunk":
        # the chunk of the mixed batch alone (no decode rows): the tensor-core
        # kernel's own roofline without the decode rows sharing the SMs
        seed = 2646
        rng = np.random.Generator(np.random.PCG64(seed))
        lens = np.array([101024], dtype=np.int32)
        pool = _pool_to_fit(lens, 0, -1)
        return Workload("prefill_chunk", seed, 64, 8, pool, "bf16", lens, np.array([1024], np.int32),
                        rng.permutation(pool),
                        description="one 1,024-token chunk over 100,000 cached tokens, alone")
    if name == "prefill_chunk_small":
        # the chunk of the small mixed batch alone: about 0.3 GB of K/V (above
        # L2), for multi-pass profiler captures of the tensor-core kernel
        seed = 2647
        rng = np.random.Generator(np.random.PCG64(seed))
        lens = np.array([41024], dtype=np.int32)
        pool = _pool_to_fit(lens, 0, -1)
        return Workload("prefill_chunk_small", seed, 64, 8, pool, "bf16", lens, np.array([1024], np.int32),
                        rng.permutation(pool),
                        description="one 1,024-token chunk over 40,000 cached tokens, alone")
    raise KeyError(name)


WORKLOADS = ("tiny", "llama8b", "llama70b_prefix", "mixed_prefill", "split_fp8")
EXTRA_WORKLOADS = ("mixed_prefill_small", "mixed_prefill_small_fp8", "mixed_prefill_fp8", "spec_verify", "spec_verify8",
                   "prefill_chunk", "prefill_chunk_small")


def small_workload(seed: int, lens, q_lens=None, hq=8, hkv=2, kv_dtype="bf16", num_blocks=None,
                   prefix_tokens=0, cow_block=-1, num_splits=0, head_dim=128, block_size=16,
                   name="small", fp8_scale_factors=None) -> Workload:
    """A small workload for parity tests: same recipe, caller-chosen sizes."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lens = np.asarray(lens, dtype=np.int32)
    if q_lens is None:
        q_lens = np.ones(len(lens), np.int32)
    if num_blocks is None:
        num_blocks = _pool_to_fit(lens, prefix_tokens, cow_block, block_size, 1.5)
    return Workload(name, seed, hq, hkv, num_blocks, kv_dtype, lens, q_lens,
                    rng.permutation(num_blocks), prefix_tokens=prefix_tokens,
                    cow_block=cow_block, num_splits=num_splits, head_dim=head_dim,
                    block_size=block_size, fp8_scale_factors=fp8_scale_factors)
