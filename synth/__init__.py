"""Seeded synthetic inputs for the paged-attention workloads.

This module is shared by both sides of every parity check (the CUDA path and
the fp64 oracle) and holds none of the attention arithmetic: it only draws
numbers.  Two kinds of randomness are used.

* Structure (sequence lengths, physical block placement) comes from numpy's
  ``Generator(PCG64(seed))`` on the host.  These arrays are small.
* Tensor values (Q, K, V) come from a counter-based generator so that any
  element can be produced on its own, on the CPU or on the GPU, with the same
  bits: ``SplitMix64`` (Steele, Lea and Flood, "Fast splittable pseudorandom
  number generators", OOPSLA 2014), whose output function is Stafford's
  "Mix13" 64-bit finaliser.  Element ``n`` of stream ``key`` is
  ``mix13(key + n * GAMMA)``.

Element ``n`` of a tensor's stream takes the three words of counters 3n, 3n+1
and 3n+2 and is the classic sum-of-twelve-uniforms approximation of a standard
normal value: the twelve 16-bit lanes of the three words are summed (an exact
integer in [0, 12 x 65535]), centred at 6 x 65535 and scaled by 2^-16 -- the
variance of twelve uniform 16-bit lanes is (65536^2 - 1) / 65536^2 x 65536^2,
so the result has mean 0 and variance 1 to within 2^-32 -- then rounded to
bf16 with round-to-nearest-even.  The centred sum is below 2^19 in magnitude,
so its conversion to fp32 and the power-of-two scaling are exact: only the
final bf16 rounding rounds.  The support is [-5.99991, 5.99991].  All of this
is integer arithmetic in torch int64 tensors (two's-complement wrap-around)
plus exact fp32 steps, so CPU and GPU produce bit-identical tensors.
"""
from __future__ import annotations

import math

import numpy as np
import torch

__all__ = [
    "MASK64", "GAMMA", "splitmix64_py", "stream_key", "mix13_t", "normal_bf16",
    "NORMAL_LANES", "NORMAL_CENTRE", "NORMAL_MAX_ABS",
]

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB

# twelve 16-bit lanes (three 64-bit words) per value
NORMAL_LANES = 12
NORMAL_CENTRE = NORMAL_LANES * 65535 // 2          # 393,210: the lanes' mean sum
# largest magnitude the generator can produce (before bf16 rounding)
NORMAL_MAX_ABS = NORMAL_CENTRE / 65536.0


def _s64(u: int) -> int:
    """Reinterpret an unsigned 64-bit integer as signed (torch int64)."""
    u &= MASK64
    return u - (1 << 64) if u >= (1 << 63) else u


def splitmix64_py(state: int) -> int:
    """Python big-int SplitMix64 output for a given (already advanced) state."""
    z = state & MASK64
    z = ((z ^ (z >> 30)) * _M1) & MASK64
    z = ((z ^ (z >> 27)) * _M2) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, tensor_id: int) -> int:
    """64-bit key of one value stream (one tensor of one workload)."""
    return splitmix64_py((seed * 0x100000001B3 + tensor_id * GAMMA + 0x1234567) & MASK64)


def _lsr(x: torch.Tensor, k: int) -> torch.Tensor:
    # logical shift right of int64 viewed as uint64
    return (x >> k) & ((1 << (64 - k)) - 1)


def mix13_t(x: torch.Tensor) -> torch.Tensor:
    """Stafford Mix13 on an int64 tensor (uint64 semantics, wrap-around)."""
    x = (x ^ _lsr(x, 30)) * _s64(_M1)
    x = (x ^ _lsr(x, 27)) * _s64(_M2)
    return x ^ _lsr(x, 31)


def normal_bf16(key: int, counters: torch.Tensor) -> torch.Tensor:
    """bf16 values with mean 0 and variance 1 (sum of twelve uniform 16-bit lanes)
    for the given int64 counters of stream ``key``.

    Works on any device; the output has the shape and device of ``counters``.
    """
    c3 = counters.to(torch.int64) * 3
    s = None
    for j in range(NORMAL_LANES // 4):
        h = mix13_t((c3 + j) * _s64(GAMMA) + _s64(key))
        part = (h & 0xFFFF) + (_lsr(h, 16) & 0xFFFF) + (_lsr(h, 32) & 0xFFFF) + _lsr(h, 48)
        s = part if s is None else s + part
    return ((s - NORMAL_CENTRE).to(torch.float32) * (2.0 ** -16)).to(torch.bfloat16)
