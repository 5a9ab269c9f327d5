"""Muon's quintic Newton-Schulz orthogonalisation in fp64 — oracle (test infrastructure only).

Source: bluscript_zero_ckpt.cpp, the ShardedMuon design note: the update is
U = NewtonSchulz(M), the iterated matrix polynomial X <- aX + (bXX' + c(XX')^2)X, where every
output entry depends on the whole matrix (hence whole-parameter ownership); the trainer's
config runs 5 steps (``muon_ns_steps``).

Readings (pages silent, listed in the design notes):
* (a, b, c) is a parameter; the default is the widely published quintic Muon triple
  (3.4445, -4.7750, 2.0315), which comes from outside the pages.
* X0 = G / (||G||_F + eps) with eps = 1e-7.
* A matrix with more rows than columns is processed as its transpose and transposed back.
"""
from __future__ import annotations

import numpy as np

DEFAULT_ABC = (3.4445, -4.7750, 2.0315)


def newton_schulz(G: np.ndarray, steps: int = 5, abc=DEFAULT_ABC, eps: float = 1e-7) -> np.ndarray:
    """fp64 Newton-Schulz of one 2-D matrix."""
    a, b, c = (float(t) for t in abc)
    X = np.asarray(G, dtype=np.float64)
    X = X / (np.linalg.norm(X) + eps)
    transposed = X.shape[0] > X.shape[1]
    if transposed:
        X = X.T
    for _ in range(steps):
        A = X @ X.T
        B = b * A + c * (A @ A)
        X = a * X + B @ X
    if transposed:
        X = X.T
    return np.ascontiguousarray(X)


def slice_block(G: np.ndarray, rows: int = 256, cols: int = 1024) -> np.ndarray:
    """The top-left block of a matrix, treated as a Newton-Schulz input of its own."""
    return np.ascontiguousarray(G[:rows, :cols])
