"""GPU parity of zopt_grad_norm_clip / zopt_clip_finalize against the oracle
(deg/zero.py grad_sq_norm; bluscript_zero_ckpt.cpp global clip block; dmuon PR #16 clip stats).

Tolerances: found_inf and clipped exact; sumsq, norm and clip_coef within 1e-6 relative
(the GPU sums fp32 runs of 8 squares into fp64, the oracle sums fp64 squares in order).
The finalize from a given sumsq is the same IEEE operation sequence on both sides, so it is
compared bit for bit.
"""
import math

import numpy as np
import pytest
import torch

from oracle import clip as OC

pytestmark = pytest.mark.gpu

SIZES = [1, 7, 8, 9, 1000, 8 * 1027 + 3, 2_000_003]


def run_norm(Z, g, max_norm, ws=None, stats=None):
    ws = Z.new_norm_workspace(g.numel()) if ws is None else ws
    stats = Z.new_clip_stats() if stats is None else stats
    Z.grad_norm_clip(g, max_norm, ws, stats)
    torch.cuda.synchronize()
    return Z.read_clip_stats(stats), ws, stats


def host_f32(g):
    return g.float().cpu().numpy()


def close(a, b, rel=1e-6):
    return abs(float(a) - float(b)) <= rel * abs(float(b)) or float(a) == float(b)


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_stats_match_oracle(zopt, n, dtype):
    gen = torch.Generator(device="cuda").manual_seed(n)
    g = (torch.randn(n, generator=gen, device="cuda") * 1e-3).to(dtype)
    for max_norm in (1.0, 1e-3, 0.0, float("inf")):
        st, _, _ = run_norm(zopt, g, max_norm)
        ref = OC.clip_stats(host_f32(g), max_norm)
        assert st["found_inf"] == ref["found_inf"] and st["clipped"] == ref["clipped"]
        assert close(st["sumsq"], ref["sumsq"]) and close(st["norm"], ref["norm"])
        assert close(st["clip_coef"], ref["clip_coef"])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("bad", [float("inf"), float("-inf"), float("nan")])
@pytest.mark.parametrize("pos", [0, 5, 8 * 999, 8 * 1027 + 2])
def test_nonfinite_sets_found_inf(zopt, dtype, bad, pos):
    n = 8 * 1027 + 3
    g = torch.full((n,), 1e-3, device="cuda", dtype=dtype)
    g[pos] = bad
    st, _, _ = run_norm(zopt, g, 1.0)
    assert st["found_inf"] and not st["clipped"] and st["clip_coef"] == 0.0


def test_extreme_finite_values(zopt):
    n = 4099
    for val, exp_inf in ((1e30, False), (3e38, True), (1e-30, False), (1e-44, False)):
        g = torch.full((n,), val, device="cuda", dtype=torch.float32)
        st, _, _ = run_norm(zopt, g, 1.0)
        ref = OC.clip_stats(host_f32(g), 1.0)
        assert st["found_inf"] == ref["found_inf"] == exp_inf, val
        if not exp_inf:
            assert close(st["sumsq"], ref["sumsq"], 1e-6), (val, st["sumsq"], ref["sumsq"])
    z = torch.zeros(10_001, device="cuda")
    st, _, _ = run_norm(zopt, z, 1.0)
    assert st["sumsq"] == 0.0 and st["norm"] == 0.0 and st["clip_coef"] == 1.0 and not st["clipped"]


def test_deterministic_and_workspace_reusable(zopt):
    g = torch.randn(3_000_017, device="cuda")
    a, ws, stats = run_norm(zopt, g, 1.0)
    for _ in range(3):
        b, _, _ = run_norm(zopt, g, 1.0, ws, stats)
        assert a == b
    # the workspace's arrival counter is back at zero
    assert int(ws[:4].view(torch.int32).item()) == 0


def test_finalize_bitwise_from_sumsq(zopt):
    rng = np.random.default_rng(0)
    stats = zopt.new_clip_stats()
    for ss in list(rng.uniform(0, 10, 50)) + [0.0, 1.0, 1e-300, 1e77, 2e77, float("inf"), float("nan")]:
        for max_norm in (1.0, 0.25, 7.0):
            raw = np.frombuffer(np.float64(ss).tobytes() + bytes(16), dtype=np.uint8).copy()
            stats.copy_(torch.from_numpy(raw))
            zopt.clip_finalize(stats, max_norm)
            st = zopt.read_clip_stats(stats)
            ref = OC.clip_from_sumsq(float(ss), max_norm)
            assert st["found_inf"] == ref["found_inf"] and st["clipped"] == ref["clipped"]
            assert np.float32(st["clip_coef"]).tobytes() == np.float32(ref["clip_coef"]).tobytes()
            if not math.isnan(ss):
                assert np.float32(st["norm"]).tobytes() == np.float32(ref["norm"]).tobytes()


def test_norm_exactly_at_max_norm(zopt):
    g = torch.zeros(64, device="cuda")
    g[3] = 1.0
    st, _, _ = run_norm(zopt, g, 1.0)
    assert st["clipped"] and st["clip_coef"] == np.float32(1.0) / np.float32(1.0 + 1e-6)
