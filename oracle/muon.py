"""Muon's update around Newton-Schulz — oracle (test infrastructure only).

Source: bluscript_zero_ckpt.cpp —
* ShardedMuon configuration: momentum 0.95, ``nesterov = true``, decoupled weight decay 0.1,
  ``ns_steps = 5``; an owner rank holds each matrix's fp32 master and momentum (8 B/element);
* the ``adjust_lr`` note: under ``match_rms_adamw`` the Newton-Schulz update's entry RMS is
  lifted to 0.2; ``original`` reproduces the modded-nanogpt scale. The quoted ratios between
  the two (4.5x for 2048x512, 21.2x for 2048x11264) are those of 0.2*sqrt(max(rows, cols))
  against sqrt(max(1, rows/cols));
* the diagnostics: ``nsratio`` = ||update||_F / sqrt(min(rows, cols)) (healthy ~1), and a
  divergence guard that rejects an update whose largest element magnitude exceeds 1000.

Readings (pages silent): the momentum is the textbook SGD form buf = mu*buf + g, with the
Nesterov update u = g + mu*buf (each operation rounded to fp32, as written); the update that
the guard and nsratio see is U = NewtonSchulz(u) before the learning-rate scale; a rejected
matrix keeps its master (its momentum has already been updated); the step is
p = p*(1 - lr*wd) - (lr*scale)*U with fp32(1 - lr*wd) and fp32(lr*scale) formed in fp64.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

from oracle.ns import DEFAULT_ABC, newton_schulz

F32 = np.float32


@dataclass(frozen=True)
class MuonHyper:
    lr: float = 8e-4
    momentum: float = 0.95
    weight_decay: float = 0.1
    nesterov: bool = True
    match_rms_adamw: bool = True
    ns_steps: int = 5
    abc: tuple = DEFAULT_ABC
    eps: float = 1e-7
    guard: float = 1000.0


def lr_scale(rows: int, cols: int, match_rms_adamw: bool) -> float:
    """The update scale: 0.2*sqrt(max(rows, cols)) (match_rms_adamw) or sqrt(max(1, rows/cols))."""
    if match_rms_adamw:
        return 0.2 * math.sqrt(max(rows, cols))
    return math.sqrt(max(1.0, rows / cols))


def momentum_f32(buf: np.ndarray, g: np.ndarray, h: MuonHyper) -> np.ndarray:
    """Updates buf in place (fp32, each operation rounded) and returns the Newton-Schulz input."""
    mu = F32(h.momentum)
    g32 = np.asarray(g, dtype=np.float32)
    buf[...] = mu * buf + g32
    return g32 + mu * buf if h.nesterov else buf.copy()


def muon_step(p: np.ndarray, buf: np.ndarray, g: np.ndarray, h: MuonHyper) -> dict:
    """One Muon step of one matrix, in place on fp32 p and buf; Newton-Schulz in fp64."""
    rows, cols = p.shape
    u = momentum_f32(buf, g, h)
    U = newton_schulz(u.astype(np.float64), steps=h.ns_steps, abc=h.abc, eps=h.eps)
    max_abs = float(np.max(np.abs(U)))
    fro = float(np.linalg.norm(U))
    rejected = not (max_abs <= h.guard)
    if not rejected:
        decay = F32(1.0 - h.lr * h.weight_decay)
        step = F32(h.lr * lr_scale(rows, cols, h.match_rms_adamw))
        p[...] = p * decay - step * U.astype(np.float32)
    return {"update": U, "fro": fro, "nsratio": fro / math.sqrt(min(rows, cols)), "max_abs": max_abs,
            "rejected": rejected}
