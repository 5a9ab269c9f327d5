"""The oracle against values the source pages print (fixtures under tests/golden/, each citing
its page and section in its header).

* bluscript_zero_ckpt.cpp: the adjust_lr ratios between the two Muon scale conventions, the
  divergence guard's threshold and the healthy nsratio;
* dmuon PR #16: the clip contract of an inf gradient;
* DeepSpeed PR #9021: how closely the one-pass rescale reproduces the directly stepped state,
  and that it needs no division by a beta.
"""
import math
import os

import numpy as np

from oracle import adamw as OA
from oracle import clip as OC
from oracle import muon as OM
from oracle.ns import newton_schulz

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def rows(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append(line.split())
    return out


def table(name):
    return {r[0]: r[1:] for r in rows(name)}


def test_adjust_lr_ratios():
    got = rows("muon_adjust_lr_ratios.txt")
    assert len(got) == 2
    for _, r, c, printed in got:
        r, c = int(r), int(c)
        ratio = OM.lr_scale(r, c, True) / OM.lr_scale(r, c, False)
        assert round(ratio, 1) == float(printed), (r, c, ratio)


def test_guard_threshold_and_healthy_nsratio():
    t = table("muon_diagnostics.txt")
    guard = float(t["guard"][0])
    assert OM.MuonHyper().guard == guard
    rng = np.random.default_rng(3)
    g = rng.normal(0, 1e-3, (128, 384)).astype(np.float32)
    p0 = rng.normal(0, 0.02, g.shape).astype(np.float32)
    # the rule at its edge: an update whose largest element equals the threshold is applied,
    # one a hair above it is rejected (its master kept)
    probe = OM.muon_step(p0.copy(), np.zeros_like(g), g, OM.MuonHyper())
    mx = probe["max_abs"]
    at = OM.MuonHyper(guard=mx)
    below = OM.MuonHyper(guard=float(np.nextafter(mx, 0.0)))
    p_at, p_below = p0.copy(), p0.copy()
    assert not OM.muon_step(p_at, np.zeros_like(g), g, at)["rejected"]
    assert OM.muon_step(p_below, np.zeros_like(g), g, below)["rejected"]
    assert np.array_equal(p_below, p0) and not np.array_equal(p_at, p0)
    # a healthy update: the quintic iteration of a Gaussian-like matrix. Five steps of the
    # default triple leave every singular value in about [0.68, 1.14], so nsratio (their RMS)
    # lies within 0.32 of the printed 1.0
    healthy = float(t["nsratio_healthy"][0])
    assert abs(probe["nsratio"] - healthy) <= 0.32
    U = newton_schulz(rng.standard_normal((256, 1024)))
    assert abs(np.linalg.norm(U) / math.sqrt(256) - healthy) <= 0.32


def test_inf_gradient_clip_contract():
    for case, coef, found, clipped in rows("clip_inf_contract.txt"):
        g = np.full(1000, 1e-3, np.float32)
        g[17] = float(case)
        st = OC.clip_stats(g, 1.0)
        assert float(st["clip_coef"]) == float(coef) and math.isfinite(float(st["clip_coef"]))
        assert bool(st["found_inf"]) == bool(int(found)) and bool(st["clipped"]) == bool(int(clipped))


def _warm(rng, n, t, h):
    p = rng.normal(0, 0.02, n)
    m = np.zeros(n)
    v = np.zeros(n)
    for s in range(1, t):
        OA.adamw_tensor_f64(p, m, v, rng.normal(0, 1e-3, n), 1.0, True, h, s)
    return p, m, v


def _rescaled_and_direct(p, m, v, g, c, h, t):
    a = [x.copy() for x in (p, m, v)]
    b = [x.copy() for x in (p, m, v)]
    OA.adamw_tensor_f32(*a, g, np.float32(1), True, OA.scalars_f32(h, t))  # the step on the old scale
    OA.rescale_step_f32(*a, g, 1.0, c, h, t)                              # re-targeted to c
    OA.adamw_tensor_f32(*b, g, np.float32(c), True, OA.scalars_f32(h, t))  # taken directly on c
    return a, b


H = OA.Hyper(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)


def test_rescale_rounding_figures():
    t = table("rescale_rounding.txt")
    rng = np.random.default_rng(12)
    # warm moments (a later step)
    p64, m64, v64 = _warm(rng, 1 << 16, 4, H)
    p, m, v = (x.astype(np.float32) for x in (p64, m64, v64))
    g = rng.normal(0, 1e-3, 1 << 16).astype(np.float32)
    a, b = _rescaled_and_direct(p, m, v, g, 0.3, H, 4)
    upd = np.max(np.abs(b[0].astype(np.float64) - p))
    w_rel = np.max(np.abs(a[0].astype(np.float64) - b[0])) / upd
    m_rel = np.max(np.abs(a[1].astype(np.float64) - b[1])) / np.max(np.abs(b[1]))
    assert 0.5 < w_rel / float(t["warm_weights_rel_update"][0]) < 2.0, w_rel
    assert 0.1 < m_rel / float(t["warm_moments_rel_max"][0]) < 10.0, m_rel
    # the first step: v's rounding grows like 2^-24 / c^2
    c = float(t["first_step_c"][0])

    def v_rel(cc):
        p1 = rng.normal(0, 0.02, 1 << 16).astype(np.float32)
        z = np.zeros_like(p1)
        g1 = rng.normal(0, 1e-3, 1 << 16).astype(np.float32)
        a1, b1 = _rescaled_and_direct(p1, z, z.copy(), g1, cc, H, 1)
        d = np.abs(a1[2].astype(np.float64) - b1[2]) / b1[2]
        return float(np.sqrt(np.mean(d * d)))

    r_c, r_10c = v_rel(c), v_rel(10 * c)
    assert 0.5 < r_c / float(t["first_step_v_rel"][0]) < 2.0, r_c
    assert 50 < r_c / r_10c < 200  # ~ c^-2
    assert r_c < 2.0 ** -24 / c ** 2


def test_rescale_needs_no_division_by_beta():
    (_, b1, b2), = rows("rescale_rounding.txt")[-1:]
    h = OA.Hyper(lr=1e-3, beta1=float(b1), beta2=float(b2), eps=1e-8, weight_decay=0.1)
    rng = np.random.default_rng(5)
    for step in (1, 3):
        p, m, v = _warm(rng, 4096, step, h)
        g = rng.normal(0, 1e-3, 4096)
        a = [x.copy() for x in (p, m, v)]
        d = [x.copy() for x in (p, m, v)]
        OA.adamw_tensor_f64(*a, g, 1.0, True, h, step)
        OA.rescale_step_f64(*a, g, 1.0, 0.25, h, step)
        OA.adamw_tensor_f64(*d, g, 0.25, True, h, step)
        assert all(np.all(np.isfinite(x)) for x in a)
        upd = np.max(np.abs(d[0] - p))
        assert np.max(np.abs(a[0] - d[0])) < 1e-9 * upd
        assert np.max(np.abs(a[1] - d[1])) <= 1e-12 * np.max(np.abs(d[1]))
