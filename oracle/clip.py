"""Gradient norm, clip coefficient, clipped / found_inf — oracle (test infrastructure only).

Sources:
* deg/zero.py, ``grad_sq_norm``: the squared L2 norm of the shard's fp32 gradient; with
  ``sim_world`` there is no all-reduce, so a simulated rank's norm is its local shard's.
* bluscript_zero_ckpt.cpp, global clip block: coef = min(1, max_norm / (norm + 1e-6));
  a non-finite norm must never reach ``min`` (NaN < 1 is false, so ``std::min`` would
  return 1 and apply no clip).
* dmuon PR #16, sync-free clip stats commit: finiteness is judged on the norm; an inf norm
  drives the coefficient to 0.0 and reports found_inf=True, clipped=False.

Readings (pages silent): the sum of squares is accumulated in fp64 over the fp32 values
(bf16 gradients promoted exactly); norm = fp32(sqrt(sumsq)); found_inf = the fp32 norm is
not finite (a NaN norm is treated like inf: coef 0, clipped False); clipped = coef < 1.
"""
from __future__ import annotations

import math

import numpy as np

F32 = np.float32


def sumsq(grad: np.ndarray) -> float:
    """sum of g**2 in fp64 over the (fp32-promoted) gradient."""
    g = np.asarray(grad, dtype=np.float32).astype(np.float64)
    return float(np.sum(g * g))


def clip_from_sumsq(ss: float, max_norm: float) -> dict:
    """The clip statistics that follow from a sum of squares.

    found_inf is judged on the fp32 norm (NaN or inf, including a finite sum whose root
    overflows fp32); then coef = 0 and clipped = False.  Otherwise
    coef = min(1, max_norm / (norm + 1e-6)) evaluated in fp32, clipped = coef < 1."""
    norm64 = math.sqrt(ss) if ss >= 0 else float("nan")
    with np.errstate(over="ignore", invalid="ignore"):
        norm = F32(norm64)
    found_inf = not math.isfinite(float(norm))
    if found_inf:
        coef = F32(0.0)
    else:
        coef = F32(max_norm) / (norm + F32(1e-6))
        if not (coef < F32(1.0)):
            coef = F32(1.0)
    return {"sumsq": ss, "norm": norm, "clip_coef": F32(coef), "clipped": bool(coef < F32(1.0)) and not found_inf,
            "found_inf": found_inf}


def clip_stats(grad: np.ndarray, max_norm: float) -> dict:
    return clip_from_sumsq(sumsq(grad), max_norm)
