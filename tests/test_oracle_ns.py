"""Pins for the oracle's Newton-Schulz (bluscript_zero_ckpt.cpp, ShardedMuon note:
X <- aX + (bXX' + c(XX')^2)X, 5 steps).

The pin is the exact closed form: with X0 = U S V', each step maps every singular value
s -> a s + b s^3 + c s^5 and keeps U and V, so NS(G) = U diag(p^k(s_i)) V'.  numpy's SVD
(a library routine that never iterates the polynomial) gives the right-hand side.
"""
import numpy as np
import pytest

from oracle.ns import DEFAULT_ABC, newton_schulz


def poly_iter(s, steps, abc):
    a, b, c = abc
    for _ in range(steps):
        s = a * s + b * s ** 3 + c * s ** 5
    return s


def svd_closed_form(G, steps=5, abc=DEFAULT_ABC, eps=1e-7):
    G = np.asarray(G, np.float64)
    U, S, Vt = np.linalg.svd(G, full_matrices=False)
    s0 = S / (np.sqrt(np.sum(S ** 2)) + eps)
    return (U * poly_iter(s0, steps, abc)) @ Vt


@pytest.mark.parametrize("shape", [(5, 7), (7, 5), (16, 17), (17, 16), (1, 8), (8, 1), (3, 3), (32, 96)])
@pytest.mark.parametrize("steps", [1, 2, 5])
def test_matches_svd_closed_form(shape, steps):
    rng = np.random.default_rng(shape[0] * 100 + shape[1] + steps)
    G = rng.standard_normal(shape)
    out = newton_schulz(G, steps=steps)
    ref = svd_closed_form(G, steps=steps)
    assert out.shape == G.shape
    assert np.linalg.norm(out - ref) <= 1e-10 * max(1.0, np.linalg.norm(ref))


def test_other_coefficients_also_match():
    rng = np.random.default_rng(9)
    G = rng.standard_normal((12, 20))
    abc = (1.875, -1.25, 0.375)  # the classical cubic-free quintic (pages silent on the triple)
    assert np.allclose(newton_schulz(G, 5, abc), svd_closed_form(G, 5, abc), atol=1e-12)


def test_row_vector_special_case():
    g = np.random.default_rng(1).standard_normal((1, 300))
    n = np.linalg.norm(g)
    s = poly_iter(n / (n + 1e-7), 5, DEFAULT_ABC)
    assert np.allclose(newton_schulz(g), s * g / n, atol=1e-13)


def test_transpose_symmetry():
    G = np.random.default_rng(2).standard_normal((40, 24))
    assert np.allclose(newton_schulz(G), newton_schulz(G.T).T, atol=1e-12)


def test_gaussian_singular_values_in_band_and_direction():
    """For a Gaussian 256x1024 input the output's singular values sit in a band around 1,
    and the output points along U V' (the orthogonal polar factor)."""
    G = np.random.default_rng(3).standard_normal((256, 1024))
    X = newton_schulz(G)
    s = np.linalg.svd(X, compute_uv=False)
    assert s.min() > 0.6 and s.max() < 1.2
    U, _, Vt = np.linalg.svd(G, full_matrices=False)
    P = U @ Vt
    cos = np.sum(X * P) / (np.linalg.norm(X) * np.linalg.norm(P))
    assert cos > 0.97
