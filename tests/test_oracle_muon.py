"""Pins for the oracle's Muon update (bluscript_zero_ckpt.cpp, ShardedMuon: momentum 0.95 with
Nesterov, adjust_lr match_rms_adamw vs original, nsratio, divergence guard)."""
import math

import numpy as np

from oracle import muon as OM
from tests.test_oracle_ns import svd_closed_form


def test_adjust_lr_ratios_printed_on_the_page():
    """The page quotes the match_rms_adamw / original ratio as 4.5x for wK/wV (2048 x 512) and
    21.2x for gate_up (2048 x 11264)."""
    r1 = OM.lr_scale(2048, 512, True) / OM.lr_scale(2048, 512, False)
    r2 = OM.lr_scale(2048, 11264, True) / OM.lr_scale(2048, 11264, False)
    assert abs(r1 - 4.5) < 0.05 and abs(r2 - 21.2) < 0.05


def test_match_rms_lifts_an_orthogonal_update_to_rms_02():
    rng = np.random.default_rng(0)
    for m, n in ((64, 256), (256, 64), (100, 100)):
        q, _ = np.linalg.qr(rng.standard_normal((max(m, n), min(m, n))))
        Q = q if m > n else q.T  # orthonormal columns (tall) or rows (wide)
        assert abs(np.sqrt(np.mean((OM.lr_scale(m, n, True) * Q) ** 2)) - 0.2) < 1e-12


def test_momentum_closed_form_and_nesterov():
    h = OM.MuonHyper(momentum=0.95)
    g = np.full(1000, 0.25, np.float32)
    buf = np.zeros(1000, np.float32)
    for k in range(1, 6):
        u = OM.momentum_f32(buf, g, h)
        geo = 0.25 * (1 - 0.95 ** k) / (1 - 0.95)
        assert np.allclose(buf, geo, rtol=4e-7)
        assert np.allclose(u, 0.25 + 0.95 * geo, rtol=4e-7)
    u_plain = OM.momentum_f32(buf.copy(), g, OM.MuonHyper(nesterov=False))
    assert np.allclose(u_plain, 0.25 * (1 - 0.95 ** 6) / (1 - 0.95), rtol=4e-7)


def test_step_against_svd_closed_form():
    """p1 = p0*(1 - lr*wd) - lr*scale*U with U from the SVD closed form of Newton-Schulz."""
    rng = np.random.default_rng(1)
    h = OM.MuonHyper(lr=8e-4)
    p = rng.normal(0, 0.02, (24, 40)).astype(np.float32)
    p0 = p.copy()
    g = rng.normal(0, 1e-3, (24, 40)).astype(np.float32)
    buf = np.zeros_like(p)
    st = OM.muon_step(p, buf, g, h)
    u = g + np.float32(0.95) * g  # buf = g after one step from zero
    U = svd_closed_form(u.astype(np.float64))
    expect = p0 * (1 - 8e-5) - 8e-4 * 0.2 * math.sqrt(40) * U
    assert np.max(np.abs(p - expect)) < 1e-8
    assert abs(st["nsratio"] - np.linalg.norm(U) / math.sqrt(24)) < 1e-9
    assert 0.5 < st["nsratio"] < 1.2 and not st["rejected"]


def test_guard_rejects_and_keeps_master():
    rng = np.random.default_rng(2)
    p = rng.normal(0, 0.02, (16, 32)).astype(np.float32)
    p0 = p.copy()
    buf = np.zeros_like(p)
    st = OM.muon_step(p, buf, rng.normal(0, 1, (16, 32)).astype(np.float32), OM.MuonHyper(guard=1e-3))
    assert st["rejected"] and np.array_equal(p, p0) and np.any(buf != 0)
