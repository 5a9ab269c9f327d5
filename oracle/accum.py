"""Micro-step gradient accumulation — oracle (test infrastructure only).

Source: deg/zero.py, ZeroMaster ``collect`` / ``reduce_scatter``: the bf16 gradients of a
step's parts are summed in fp32 (the first part is taken as is, later parts are added), and
``grad_sq_norm`` reads the finished fp32 sum.

Reading (pages silent on the order): parts are added in the order they arrive, each addition
rounded to fp32: acc = ((g1 + g2) + g3) + ...
"""
from __future__ import annotations

import numpy as np


def accumulate(parts: list) -> np.ndarray:
    """fp32 sum of the parts (each promoted exactly to fp32), in order."""
    acc = np.asarray(parts[0], dtype=np.float32).copy()
    for g in parts[1:]:
        acc = acc + np.asarray(g, dtype=np.float32)
    return acc
