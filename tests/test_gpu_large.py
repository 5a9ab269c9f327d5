"""A shard longer than 2^31 elements: the element-wise kernels (norm, AdamW, rescale,
accumulation) index with 64-bit integers.

n = 2^31 + 4099 elements (~35 GB of fp32 master, moments and bf16 gradient and weights on the
device). The inputs repeat with a period of L = 4096 elements and every output element depends
on its own inputs only (plus the clip coefficient), so every output is periodic too. The whole
output is checked, on the GPU, against the oracle's result for one period; the ragged tail
(n mod L = 3) against the period's first elements. The sum of squares has the closed form
(n div L) * sum(period^2) + sum(first tail^2).
"""
import math

import numpy as np
import pytest
import torch

from oracle import adamw as OA
from oracle import clip as OC
from oracle.accum import accumulate
from oracle.bf16 import f32_to_bf16_bits

pytestmark = pytest.mark.gpu

N = (1 << 31) + 4099
L = 4096
FULL, TAIL = N // L, N % L


def periodic(pattern, device="cuda"):
    """The pattern repeated to N elements, on the device."""
    return pattern.to(device).repeat(FULL + 1)[:N]


def assert_periodic(t, expect_bits):
    """t (4-byte or 2-byte elements) equals the expected period bit for bit everywhere."""
    it = torch.int32 if t.element_size() == 4 else torch.int16
    bits = t.view(it)
    want = torch.from_numpy(expect_bits.astype(np.int32 if it == torch.int32 else np.int16)).to(t.device)
    assert bool((bits[:FULL * L].view(FULL, L) == want[None, :]).all())
    assert torch.equal(bits[FULL * L:], want[:TAIL])


def closed_form_sumsq(x):
    """Sum of squares of the periodic vector built from the float period x: the squares are
    exact in fp64 and math.fsum adds them correctly rounded, so the result is within a few
    fp64 ulps of the exact sum."""
    sq = [float(v) * float(v) for v in x.astype(np.float64)]
    return math.fsum([FULL * math.fsum(sq), math.fsum(sq[:TAIL])])


def test_adamw_step_and_norm_past_2_to_the_31(zopt):
    rng = np.random.default_rng(2031)
    g_pat = torch.from_numpy(rng.normal(0, 1e-3, L).astype(np.float32)).to(torch.bfloat16)
    p_pat = rng.normal(0, 0.02, L).astype(np.float32)
    lay = zopt.ShardLayout([N], [True], 1 << 25, 1, 0)
    assert lay.shard_len == N
    g = periodic(g_pat)
    p = periodic(torch.from_numpy(p_pat))
    m = torch.zeros(N, device="cuda")
    v = torch.zeros(N, device="cuda")
    out = torch.empty(N, dtype=torch.int16, device="cuda")
    ws, clip, state = zopt.new_norm_workspace(N), zopt.new_clip_stats(), zopt.new_adam_state()
    h = OA.Hyper(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
    max_norm = 0.05
    zopt.grad_norm_clip(g, max_norm, ws, clip)
    zopt.adamw_step(lay, lay.device_table(), p, m, v, g, out, lr=h.lr, beta1=h.beta1, beta2=h.beta2, eps=h.eps,
                    weight_decay=h.weight_decay, clip_stats=clip, adam_state=state)
    torch.cuda.synchronize()
    st = zopt.read_clip_stats(clip)
    g_np = g_pat.float().numpy()
    ss = closed_form_sumsq(g_np)
    assert abs(st["sumsq"] - ss) <= 1e-6 * ss
    ref = OC.clip_from_sumsq(ss, max_norm)
    assert abs(float(st["clip_coef"]) - float(ref["clip_coef"])) <= 1e-6 * float(ref["clip_coef"])
    assert not st["found_inf"] and st["clipped"] and ref["clipped"]
    # one period through the oracle with the GPU's coefficient (t = 1, fresh moments)
    pe, me, ve = p_pat.copy(), np.zeros(L, np.float32), np.zeros(L, np.float32)
    OA.adamw_tensor_f32(pe, me, ve, g_np, np.float32(st["clip_coef"]), True, OA.scalars_f32(h, 1))
    for t, e in ((p, pe), (m, me), (v, ve)):
        assert_periodic(t, e.view(np.int32))
    assert_periodic(out, f32_to_bf16_bits(pe).view(np.int16))
    assert zopt.read_adam_state(state)["step"] == 1
    # the same step re-targeted to half the coefficient, in one pass over the whole shard
    coef = float(st["clip_coef"])
    zopt.adamw_rescale_step(lay, p, m, v, g, out, lr=h.lr, old_scale=coef, new_scale=coef / 2, beta1=h.beta1,
                            beta2=h.beta2, eps=h.eps, weight_decay=h.weight_decay, adam_state=state)
    torch.cuda.synchronize()
    OA.rescale_step_f32(pe, me, ve, g_np, coef, coef / 2, h, 1)
    for t, e in ((p, pe), (m, me), (v, ve)):
        assert_periodic(t, e.view(np.int32))
    assert_periodic(out, f32_to_bf16_bits(pe).view(np.int16))
    del g, p, m, v, out
    torch.cuda.empty_cache()


def test_accumulation_past_2_to_the_31(zopt):
    rng = np.random.default_rng(2032)
    pats = [torch.from_numpy(rng.normal(0, 1e-3, L).astype(np.float32)).to(torch.bfloat16) for _ in range(2)]
    acc = torch.empty(N, device="cuda")
    ws, clip = zopt.new_norm_workspace(N), zopt.new_clip_stats()
    for k, pat in enumerate(pats):
        micro = periodic(pat)
        zopt.grad_accumulate(acc, micro, first=k == 0, last=k == len(pats) - 1, max_norm=1.0, ws=ws, stats=clip)
        torch.cuda.synchronize()
        del micro
    want = accumulate([pat.float().numpy() for pat in pats])
    assert_periodic(acc, want.view(np.int32))
    ss = closed_form_sumsq(want)
    st = zopt.read_clip_stats(clip)
    assert abs(st["sumsq"] - ss) <= 1e-6 * ss
    del acc
    torch.cuda.empty_cache()
