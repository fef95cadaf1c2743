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

The 64-bit word is turned into an approximately standard-normal value with an
exact Irwin-Hall(4) construction: the four 16-bit lanes are summed (an exact
integer), centred, converted to fp32 (exact, |x| < 2^18) and multiplied once by
the fp32 constant sqrt(3)/65536 (one IEEE multiply: identical on every IEEE
machine), then rounded to bf16 with round-to-nearest-even.  The result has
mean 0, variance 1 and support [-3.4641, 3.4641].  All of this is integer
arithmetic in torch int64 tensors (two's-complement wrap-around) plus one fp32
multiply, so CPU and GPU produce bit-identical tensors.
"""
from __future__ import annotations

import math

import numpy as np
import torch

__all__ = [
    "MASK64", "GAMMA", "splitmix64_py", "stream_key", "mix13_t", "normal_bf16",
    "IH4_SCALE_F32", "IH4_MAX_ABS",
]

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB

# fp32(sqrt(3) / 65536): one Irwin-Hall(4) unit of 16-bit lanes -> unit variance
IH4_SCALE_F32 = np.float32(math.sqrt(3.0) / 65536.0)
# largest magnitude the generator can produce (before bf16 rounding)
IH4_MAX_ABS = float(np.float32(np.float32(131070.0) * IH4_SCALE_F32))


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
    """bf16 N(0,1)-like values for the given int64 counters of stream ``key``.

    Works on any device; the output has the shape and device of ``counters``.
    """
    dev = counters.device
    x = counters.to(torch.int64) * _s64(GAMMA) + _s64(key)
    h = mix13_t(x)
    s = (h & 0xFFFF) + (_lsr(h, 16) & 0xFFFF) + (_lsr(h, 32) & 0xFFFF) + _lsr(h, 48)
    c = torch.tensor(float(IH4_SCALE_F32), dtype=torch.float32, device=dev)
    f = (s - 131070).to(torch.float32) * c
    return f.to(torch.bfloat16)
