"""Pins for the oracle's AdamW (dmuon PR #16 foreach-AdamW op order; DeepSpeed PR #9021
grad_scale on load; deg/zero.py flat == per-tensor; bluscript_zero_ckpt.cpp ZeroConfig).

Each pin is something other than the oracle itself: the first-step closed form
(m_hat = g, v_hat = g^2), torch.optim.AdamW (an independent library implementation),
math.pow, invariants the pages state (flat == per-tensor bitwise; a pre-scaled gradient
== grad_scale on load, bitwise).
"""
import math

import numpy as np
import pytest
import torch

from oracle import adamw as OA
from oracle import layout as OL

H = OA.Hyper(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)


def test_beta_power_against_math_pow():
    for beta in (0.9, 0.95, 0.999, 0.5, 0.0, 1.0):
        for t in list(range(0, 70)) + [1000, 12345, 2 ** 20 + 7]:
            got = OA.beta_power(beta, t)
            ref = math.pow(beta, t)
            # squaring doubles the relative error, so both methods carry about t units of
            # 2^-53 of relative error: bound by (2t + 8) of them
            assert abs(got - ref) <= (2 * t + 8) * 2.0 ** -53 * ref or got == ref, (beta, t)
    # and against the repeated product for small t (a different order of the same multiplies)
    for t in range(1, 40):
        prod = 1.0
        for _ in range(t):
            prod *= 0.95
        assert abs(OA.beta_power(0.95, t) - prod) <= (3 * t + 8) * 2.0 ** -53 * prod


def rand_tensors(rng, shapes):
    ps = [rng.normal(0, 0.02, s).astype(np.float32) if len(s) == 2 else np.ones(s, np.float32) for s in shapes]
    return ps


def test_first_step_closed_form_f64():
    rng = np.random.default_rng(0)
    p0 = rng.normal(0, 0.02, 1000)
    g = rng.normal(0, 1e-3, 1000)
    p, m, v = p0.copy(), np.zeros(1000), np.zeros(1000)
    OA.adamw_tensor_f64(p, m, v, g, 1.0, True, H, 1)
    expect = p0 * (1 - H.lr * H.weight_decay) - H.lr * g / (np.abs(g) + H.eps)
    assert np.max(np.abs(p - expect) / np.abs(expect)) < 1e-10
    assert np.allclose(m, (1 - H.beta1) * g, rtol=1e-15, atol=0)
    assert np.allclose(v, (1 - H.beta2) * g * g, rtol=1e-15, atol=0)


def test_first_step_closed_form_f32():
    rng = np.random.default_rng(1)
    p0 = rng.normal(0, 0.02, 4096).astype(np.float32)
    g = rng.normal(0, 1e-3, 4096).astype(np.float32)
    p, m, v = p0.copy(), np.zeros(4096, np.float32), np.zeros(4096, np.float32)
    OA.adamw_tensor_f32(p, m, v, g, np.float32(1), True, OA.scalars_f32(H, 1))
    expect = p0.astype(np.float64) * (1 - H.lr * H.weight_decay) - H.lr * g / (np.abs(g.astype(np.float64)) + H.eps)
    # a few fp32 roundings of a value of size |p| + lr
    assert np.max(np.abs(p - expect)) < 8 * np.finfo(np.float32).eps * (np.max(np.abs(p0)) + H.lr)


def test_zero_grad_first_step_only_decays():
    p0 = np.linspace(-1, 1, 33, dtype=np.float32)
    p, m, v = p0.copy(), np.zeros(33, np.float32), np.zeros(33, np.float32)
    sc = OA.scalars_f32(H, 1)
    OA.adamw_tensor_f32(p, m, v, np.zeros(33, np.float32), np.float32(1), True, sc)
    assert np.array_equal(p, p0 * sc.decay)
    p2 = p0.copy()
    OA.adamw_tensor_f32(p2, m * 0, v * 0, np.zeros(33, np.float32), np.float32(1), False, sc)
    assert np.array_equal(p2, p0)


def test_against_torch_adamw():
    """torch.optim.AdamW (single-tensor path, fp32) as an independent implementation."""
    rng = np.random.default_rng(2)
    shapes = [(64, 32), (32,), (48, 16), (7,)]
    ps = rand_tensors(rng, shapes)
    tps = [torch.nn.Parameter(torch.from_numpy(p.copy())) for p in ps]
    groups = [{"params": [t for t, s in zip(tps, shapes) if len(s) == 2], "weight_decay": H.weight_decay},
              {"params": [t for t, s in zip(tps, shapes) if len(s) == 1], "weight_decay": 0.0}]
    opt = torch.optim.AdamW(groups, lr=H.lr, betas=(H.beta1, H.beta2), eps=H.eps, foreach=False)
    ms = [np.zeros_like(p) for p in ps]
    vs = [np.zeros_like(p) for p in ps]
    for t in range(1, 6):
        gs = [rng.normal(0, 1e-3, s).astype(np.float32) for s in shapes]
        for tp, g in zip(tps, gs):
            tp.grad = torch.from_numpy(g.copy())
        opt.step()
        OA.step_tensors(ps, ms, vs, gs, [len(s) == 2 for s in shapes], 1.0, H, t)
    for p, tp, m, v in zip(ps, tps, ms, vs):
        st = opt.state[tp]
        assert np.allclose(p, tp.detach().numpy(), rtol=2e-6, atol=1e-9)
        # torch forms m by lerp, so where beta1*m and (1-beta1)*g nearly cancel the two
        # roundings differ: compare against the moment's own scale
        tm, tv = st["exp_avg"].numpy(), st["exp_avg_sq"].numpy()
        assert np.max(np.abs(m - tm)) <= 1e-6 * np.max(np.abs(tm))
        assert np.max(np.abs(v - tv)) <= 1e-6 * np.max(np.abs(tv))


def test_f32_tracks_f64_over_ten_steps():
    rng = np.random.default_rng(3)
    p32 = rng.normal(0, 0.02, 5000).astype(np.float32)
    p64 = p32.astype(np.float64)
    m32, v32 = np.zeros_like(p32), np.zeros_like(p32)
    m64, v64 = np.zeros_like(p64), np.zeros_like(p64)
    sc_step = 0
    for t in range(1, 11):
        g = rng.normal(0, 1e-3, 5000).astype(np.float32)
        OA.adamw_tensor_f32(p32, m32, v32, g, np.float32(1), True, OA.scalars_f32(H, t))
        OA.adamw_tensor_f64(p64, m64, v64, g, 1.0, True, H, t)
        sc_step = t
    assert sc_step == 10
    # elements that pass near zero have no useful relative error; bound the absolute one
    assert np.max(np.abs(p32 - p64)) < 1e-6 * (np.max(np.abs(p64)) + 10 * H.lr)


def test_flat_equals_per_tensor_bitwise():
    """Element-wise AdamW over the flat shard is the same arithmetic as per tensor."""
    rng = np.random.default_rng(4)
    shapes = [(33, 7), (5,), (64, 3), (1,), (9, 9)]
    numel = [int(np.prod(s)) for s in shapes]
    decay = [len(s) == 2 for s in shapes]
    ps = [p.reshape(-1) for p in rand_tensors(rng, shapes)]
    ms = [np.zeros_like(p) for p in ps]
    vs = [np.zeros_like(p) for p in ps]
    for world in (1, 3, 8):
        for rank in range(world):
            flat_p = np.concatenate(ps)
            sp = OL.gather_shard(flat_p, numel, 16, world, rank)
            sm = np.zeros_like(sp)
            sv = np.zeros_like(sp)
            mask = OL.decay_mask_of_shard(decay, numel, 16, world, rank)
            tp = [p.copy() for p in ps]
            tm = [m.copy() for m in ms]
            tv = [v.copy() for v in vs]
            for t in range(1, 4):
                gs = [rng.normal(0, 1e-3, n).astype(np.float32) for n in numel]
                coef = np.float32(0.75)
                OA.step_tensors(tp, tm, tv, gs, decay, coef, H, t)
                sg = OL.gather_shard(np.concatenate(gs), numel, 16, world, rank)
                OA.step_flat_f32(sp, sm, sv, sg, mask, coef, H, t)
                for a, b in ((sp, tp), (sm, tm), (sv, tv)):
                    ref = OL.gather_shard(np.concatenate(b), numel, 16, world, rank)
                    assert np.array_equal(a.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("n", [1, 7, 8, 9, 1027])
def test_grad_scale_on_load_equals_prescaled(n):
    """grad_scale applied on load == the gradient scaled beforehand, bit for bit, 3 steps."""
    rng = np.random.default_rng(5 + n)
    pa = rng.normal(0, 0.02, n).astype(np.float32)
    pb = pa.copy()
    ma, va, mb, vb = (np.zeros(n, np.float32) for _ in range(4))
    scale = np.float32(0.3141)
    for t in range(1, 4):
        g = rng.normal(0, 1e-3, n).astype(np.float32)
        sc = OA.scalars_f32(H, t)
        OA.adamw_tensor_f32(pa, ma, va, g, scale, True, sc)
        OA.adamw_tensor_f32(pb, mb, vb, g * scale, np.float32(1), True, sc)
    assert np.array_equal(pa.view(np.uint32), pb.view(np.uint32))
    assert np.array_equal(va.view(np.uint32), vb.view(np.uint32))


def test_bf16_grad_equals_its_fp32_promotion():
    """A bf16 gradient steps exactly as its fp32 promotion (torch's widening as the pin)."""
    from oracle.bf16 import bf16_bits_to_f32
    rng = np.random.default_rng(6)
    g16 = torch.from_numpy(rng.normal(0, 1e-3, 999).astype(np.float32)).to(torch.bfloat16)
    via_oracle = bf16_bits_to_f32(g16.view(torch.int16).numpy().view(np.uint16))
    via_torch = g16.to(torch.float32).numpy()
    assert np.array_equal(via_oracle, via_torch)
    pa = rng.normal(0, 0.02, 999).astype(np.float32)
    pb = pa.copy()
    z = [np.zeros(999, np.float32) for _ in range(4)]
    sc = OA.scalars_f32(H, 1)
    OA.adamw_tensor_f32(pa, z[0], z[1], via_oracle, np.float32(1), True, sc)
    OA.adamw_tensor_f32(pb, z[2], z[3], via_torch, np.float32(1), True, sc)
    assert np.array_equal(pa, pb)


def test_scalars_are_fp64_rounded_once():
    sc = OA.scalars_f32(H, 1)
    assert sc.one_minus_beta1 == np.float32(1.0 - 0.9)
    assert sc.one_minus_beta1 != np.float32(1.0) - np.float32(0.9)  # the reading matters
    assert sc.step_size == np.float32(1e-3 / (1.0 - 0.9))
    assert sc.bc2_sqrt == np.float32(math.sqrt(1.0 - 0.95))
    assert sc.decay == np.float32(1.0 - 1e-4)


def _warm(rng, n, t):
    p = rng.normal(0, 0.02, n)
    m = np.zeros(n)
    v = np.zeros(n)
    for s in range(1, t):
        OA.adamw_tensor_f64(p, m, v, rng.normal(0, 1e-3, n), 1.0, True, H, s)
    return p, m, v


def test_rescale_equals_direct_step_in_fp64():
    """DeepSpeed PR #9021: the rescaled state is the state of the step taken directly on the new
    scale (here in fp64, up to fp64 rounding)."""
    rng = np.random.default_rng(11)
    for t in (1, 5):
        p, m, v = _warm(rng, 2000, t)
        g = rng.normal(0, 1e-3, 2000)
        a = [x.copy() for x in (p, m, v)]
        b = [x.copy() for x in (p, m, v)]
        OA.adamw_tensor_f64(*a, g, 1.0, True, H, t)           # speculative step on the old scale
        OA.rescale_step_f64(*a, g, 1.0, 0.3, H, t)            # re-targeted to 0.3
        OA.adamw_tensor_f64(*b, g, 0.3, True, H, t)           # the step taken directly on 0.3
        upd = np.max(np.abs(b[0] - p))
        assert np.max(np.abs(a[0] - b[0])) < 1e-9 * upd
        assert np.max(np.abs(a[1] - b[1])) < 1e-12 * np.max(np.abs(b[1]))
        assert np.max(np.abs(a[2] - b[2])) < 1e-9 * np.max(np.abs(b[2]))


def test_rescale_f32_close_to_direct_and_same_scale_is_bitwise():
    rng = np.random.default_rng(12)
    p64, m64, v64 = _warm(rng, 4096, 4)
    p, m, v = (x.astype(np.float32) for x in (p64, m64, v64))
    g = rng.normal(0, 1e-3, 4096).astype(np.float32)
    a = [x.copy() for x in (p, m, v)]
    b = [x.copy() for x in (p, m, v)]
    OA.adamw_tensor_f32(*a, g, np.float32(1), True, OA.scalars_f32(H, 4))
    c = [x.copy() for x in a]
    OA.rescale_step_f32(*c, g, 1.0, 1.0, H, 4)  # to the same scale: moments bit for bit, p too
    for x, y in zip(a, c):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))
    OA.rescale_step_f32(*a, g, 1.0, 0.5, H, 4)
    OA.adamw_tensor_f32(*b, g, np.float32(0.5), True, OA.scalars_f32(H, 4))
    upd = np.max(np.abs(b[0] - p))
    assert np.max(np.abs(a[0] - b[0])) < 1e-4 * upd  # the page measures 7.5e-6 of the update
    assert np.max(np.abs(a[1] - b[1])) < 1e-6 * np.max(np.abs(b[1]))


def test_rescale_keeps_nan_in_v():
    p, m, v = (np.ones(4, np.float32) for _ in range(3))
    v[1] = np.nan
    OA.rescale_step_f32(p, m, v, np.ones(4, np.float32), 1.0, 0.0, H, 3)
    assert np.isnan(v[1]) and np.all(v[[0, 2, 3]] >= 0)
