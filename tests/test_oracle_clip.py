"""Pins for the oracle's norm / clip / found_inf (deg/zero.py grad_sq_norm;
bluscript_zero_ckpt.cpp global clip block; dmuon PR #16 sync-free clip stats).

Pinned by closed forms (constant and one-hot gradients), exact summation (math.fsum),
torch.nn.utils.clip_grad_norm_ (an independent library routine using the same
1e-6-guarded coefficient), and the inf/NaN contract the pages state.
"""
import math

import numpy as np
import torch

from oracle import clip as OC

F32 = np.float32


def test_constant_grad_closed_form():
    g = np.full(1000, 0.5, np.float32)
    st = OC.clip_stats(g, 1.0)
    assert st["sumsq"] == 1000 * 0.25
    assert st["norm"] == F32(math.sqrt(250.0))
    assert st["clip_coef"] == F32(1.0) / (F32(math.sqrt(250.0)) + F32(1e-6))
    assert st["clipped"] and not st["found_inf"]


def test_one_hot_norm_is_abs_value():
    g = np.zeros(77, np.float32)
    g[13] = -3.0
    st = OC.clip_stats(g, 10.0)
    assert st["norm"] == F32(3.0)
    assert st["clip_coef"] == F32(1.0) and not st["clipped"]


def test_inf_and_nan_set_found_inf_not_clipped():
    for bad in (np.inf, -np.inf, np.nan):
        g = np.ones(10, np.float32)
        g[4] = bad
        st = OC.clip_stats(g, 1.0)
        assert st["found_inf"] and not st["clipped"] and st["clip_coef"] == 0.0


def test_huge_finite_values_are_not_inf():
    g = np.full(8, 1e30, np.float32)
    st = OC.clip_stats(g, 1.0)
    assert not st["found_inf"] and st["clipped"]
    assert math.isclose(float(st["norm"]), math.sqrt(8) * 1e30, rel_tol=1e-7)


def test_norm_exactly_max_norm_still_clips():
    """coef = 1/(1 + 1e-6f) < 1, so a norm of exactly max_norm counts as clipped."""
    g = np.zeros(4, np.float32)
    g[0] = 1.0
    st = OC.clip_stats(g, 1.0)
    assert st["clip_coef"] == F32(1.0) / F32(1.0 + 1e-6) and st["clip_coef"] < 1 and st["clipped"]
    # just below the boundary: max_norm slightly larger than norm + 1e-6 -> no clip
    st2 = OC.clip_stats(g, float(np.nextafter(F32(1.0) + F32(1e-6), F32(2.0))))
    assert st2["clip_coef"] == F32(1.0) and not st2["clipped"]


def test_sumsq_against_exact_fsum():
    rng = np.random.default_rng(0)
    g = rng.normal(0, 1e-3, 100_003).astype(np.float32)
    exact = math.fsum(float(x) * float(x) for x in g.astype(np.float64))
    assert abs(OC.sumsq(g) - exact) <= 1e-13 * exact


def test_against_torch_clip_grad_norm():
    rng = np.random.default_rng(1)
    gs = [rng.normal(0, 0.3, n).astype(np.float32) for n in (1000, 37, 4096)]
    ps = [torch.nn.Parameter(torch.zeros(len(g))) for g in gs]
    for p, g in zip(ps, gs):
        p.grad = torch.from_numpy(g.copy())
    total = torch.nn.utils.clip_grad_norm_(ps, max_norm=1.0)
    st = OC.clip_stats(np.concatenate(gs), 1.0)
    assert math.isclose(float(total), float(st["norm"]), rel_tol=2e-7)
    # torch scaled the grads in place by its coefficient; recover it from one element
    coef_torch = ps[0].grad[0].item() / gs[0][0]
    assert math.isclose(coef_torch, float(st["clip_coef"]), rel_tol=1e-6)
