"""fp32 -> bf16 round-to-nearest-even — oracle (test infrastructure only).

Source: deg/zero.py, ``gather_params`` ("rounds each rank's updated shard to bf16": the
shard cast to the compute dtype, bitwise what the unsharded ``p.copy_(master)`` gives).
The rounding is IEEE round-to-nearest, ties to even, on the top 16 bits of the fp32
pattern; NaN stays a (quiet) NaN with its sign; values that round past the largest finite
bf16 become infinity, as RNE requires.
"""
from __future__ import annotations

import numpy as np


def f32_to_bf16_bits(x) -> np.ndarray:
    """bf16 bit patterns (uint16) of fp32 values, round-to-nearest-even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    exp_all_ones = (u & 0x7F800000) == 0x7F800000
    mant_nonzero = (u & 0x007FFFFF) != 0
    is_nan = exp_all_ones & mant_nonzero
    lsb = (u >> 16) & 1
    rounded = (u + 0x7FFF + lsb) >> 16
    quiet_nan = ((u >> 16) & 0x8000) | 0x7FC0
    out = np.where(is_nan, quiet_nan, rounded)
    return out.astype(np.uint16)


def bf16_bits_to_f32(b) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32 values."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
