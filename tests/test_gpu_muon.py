"""GPU parity of zopt_muon_step against the oracle's Muon update (bluscript_zero_ckpt.cpp,
ShardedMuon: momentum with Nesterov, U = NewtonSchulz(u), adjust_lr scale, decoupled decay,
nsratio and the divergence guard).

Bar: the momentum buffer bit for bit (fp32, same operation order); the applied update
(p_old*fp32(1 - lr*wd) - p_new) / fp32(lr*scale) within relative Frobenius error 2e-2 of the
oracle's fp64 Newton-Schulz of the same u (the bf16 Newton-Schulz tolerance); nsratio within
2e-2; the bf16 weights bit for bit the round-out of the new master; a rejected matrix keeps
its master bit for bit.
"""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import muon as OM
from oracle.bf16 import f32_to_bf16_bits
from oracle.ns import newton_schulz

pytestmark = pytest.mark.gpu


def rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


@pytest.mark.parametrize("rows,cols,batch,group", [(256, 768, 1, 1), (768, 256, 1, 1), (384, 1000, 3, 2),
                                                    (2048, 512, 2, 2), (130, 70, 1, 1)])
@pytest.mark.parametrize("match", [True, False])
def test_three_steps_match_oracle(zopt, rows, cols, batch, group, match):
    h = OM.MuonHyper(lr=8e-4, match_rms_adamw=match)
    gen = torch.Generator(device="cuda").manual_seed(rows + cols + batch)
    p = (torch.randn(batch, rows, cols, generator=gen, device="cuda") * 0.02)
    buf = torch.zeros_like(p)
    out = torch.zeros(batch, rows, cols, dtype=torch.int16, device="cuda")
    ws = zopt.new_muon_workspace(rows, cols, group)
    stats = zopt.new_muon_stats(batch)
    ref_buf = np.zeros((batch, rows, cols), np.float32)
    decay = np.float32(1.0 - h.lr * h.weight_decay)
    step = np.float32(h.lr * OM.lr_scale(rows, cols, match))
    for s in range(3):
        g = (torch.randn(batch, rows, cols, generator=gen, device="cuda") * 1e-3).bfloat16()
        p_old = p.cpu().numpy()
        zopt.muon_step(p, buf, g, out, ws, stats, lr=h.lr, match_rms_adamw=match)
        torch.cuda.synchronize()
        st = zopt.read_muon_stats(stats)
        pn = p.cpu().numpy()
        for b in range(batch):
            u = OM.momentum_f32(ref_buf[b], g[b].float().cpu().numpy(), h)
            U_ref = newton_schulz(u.astype(np.float64), steps=5)
            applied = (p_old[b] * decay - pn[b]).astype(np.float64) / float(step)
            assert rel(applied, U_ref) <= 2e-2, (s, b)
            assert abs(st[b]["ns_ratio"] - np.linalg.norm(U_ref) / math.sqrt(min(rows, cols))) <= 2e-2
            assert not st[b]["rejected"] and abs(st[b]["max_abs"] / np.max(np.abs(U_ref)) - 1) < 0.1
        assert np.array_equal(buf.cpu().numpy().view(np.uint32), ref_buf.view(np.uint32))
        assert np.array_equal(out.cpu().numpy().view(np.uint16), f32_to_bf16_bits(pn))


def test_guard_rejects_keeps_master_updates_momentum(zopt):
    rows, cols = 200, 300
    p = torch.randn(rows, cols, device="cuda") * 0.02
    p0 = p.clone()
    buf = torch.zeros_like(p)
    g = torch.randn(rows, cols, device="cuda")
    out = torch.zeros(rows, cols, dtype=torch.int16, device="cuda")
    stats = zopt.new_muon_stats()
    zopt.muon_step(p, buf, g, out, zopt.new_muon_workspace(rows, cols), stats, lr=1e-3, guard=1e-3)
    torch.cuda.synchronize()
    st = zopt.read_muon_stats(stats)[0]
    assert st["rejected"] and torch.equal(p, p0) and torch.equal(buf, g)
    assert np.array_equal(out.cpu().numpy().view(np.uint16), f32_to_bf16_bits(p0.cpu().numpy()))


def run_muon_set(Z, params, seed, steps, lr_at, zero_row_frac=0.0):
    """Steps a parameter set's Muon matrices ``steps`` times, one zopt_muon_step_many call per step
    over the set's shapes (each shape's matrices one batch, as a trainer groups them), and checks
    every matrix after every step against the oracle: the momentum buffer bit for bit (carried by
    the oracle from zero), the applied update within 2e-2 of the fp64 Newton-Schulz of the oracle's
    u, no rejection, and the bf16 weights bit for bit the new master's. The learning rate of 0-based
    step s is lr_at(s). Inputs: workloads' masters (N(0, 0.02)) and bf16 gradients (N(0, 1e-3),
    a seeded fraction of zero rows)."""
    shapes = []
    for prm in params:
        if prm.shape not in shapes:
            shapes.append(prm.shape)
    groups = [[i for i, prm in enumerate(params) if prm.shape == sh] for sh in shapes]
    master = [torch.stack([workloads.master_for(params[i], seed, 20_000 + i) for i in idx]).cuda() for idx in groups]
    buf = [torch.zeros_like(x) for x in master]
    out = [torch.zeros(x.shape, dtype=torch.int16, device="cuda") for x in master]
    stats = [Z.new_muon_stats(len(idx)) for idx in groups]
    ws = Z.new_muon_workspace_many([(r, c, len(idx)) for (r, c), idx in zip(shapes, groups)])
    ref_buf = [np.zeros(tuple(x.shape), np.float32) for x in master]
    for s in range(steps):
        lr = lr_at(s)
        h = OM.MuonHyper(lr=lr)
        grads = [torch.stack([workloads.grad_for(params[i], seed, 300_000 + 1000 * s + i, zero_row_frac)
                              for i in idx]) for idx in groups]
        p_old = [x.cpu().numpy() for x in master]
        Z.muon_step_many([(master[k], buf[k], grads[k].cuda(), out[k], stats[k]) for k in range(len(groups))], ws,
                         lr=lr)
        torch.cuda.synchronize()
        decay = np.float32(1.0 - lr * h.weight_decay)
        for k, (r, c) in enumerate(shapes):
            step = np.float32(lr * OM.lr_scale(r, c, h.match_rms_adamw))
            pn = master[k].cpu().numpy()
            st = Z.read_muon_stats(stats[k])
            g_np = grads[k].float().numpy()
            for b in range(len(groups[k])):
                u = OM.momentum_f32(ref_buf[k][b], g_np[b], h)
                U_ref = newton_schulz(u.astype(np.float64), steps=h.ns_steps)
                applied = (p_old[k][b] * decay - pn[b]).astype(np.float64) / float(step)
                assert rel(applied, U_ref) <= 2e-2, (s, (r, c), b)
                assert not st[b]["rejected"]
            assert np.array_equal(buf[k].cpu().numpy().view(np.uint32), ref_buf[k].view(np.uint32)), (s, (r, c))
            assert np.array_equal(out[k].cpu().numpy().view(np.uint16), f32_to_bf16_bits(pn)), (s, (r, c))


def test_gpt2_body_ten_wsd_steps(zopt):
    """The GPT-2-small body's 48 Muon matrices (768x2304, 768x768, 768x3072, 3072x768; 1 % zero
    gradient rows) through the set's ten stated steps, on the WSD curve the AdamW group follows
    with Muon's own peak and floor (8e-4, 8e-5; bluscript_zero_ckpt.cpp feeds both groups one
    schedule): the decay phase's learning rates reach the update."""
    w = workloads.get("c2")
    lrs = [w.muon_lr_at(s) for s in range(w.steps)]
    assert w.steps == 10 and len(w.muon) == 48 and lrs[9] == 8e-5 and lrs[8] < lrs[7] < lrs[6] == 8e-4
    run_muon_set(zopt, w.muon, w.seed, w.steps, w.muon_lr_at, w.zero_row_frac)


def test_llama_owned_set_five_steps(zopt):
    """The 1.1B set's matrices owned by rank 0 of 8 (round-robin: 4 x Wq 2048^2, 4 x Wv 2048x512,
    4 x gate_up 2048x11264) through the set's five stated steps in one call per step, as the
    benchmark's Muon step runs them."""
    w = workloads.get("c3")
    owned = w.owned_muon()
    assert len(owned) == 12 and w.steps == 5
    run_muon_set(zopt, owned, w.seed, w.steps, w.muon_lr_at)


def test_many_shapes_equal_single_calls(zopt):
    """zopt_muon_step_many over several shapes (bf16 and fp32 gradients, with and without the
    bf16 round-out, a tall matrix, a CTA-pair size) for two steps: master, momentum, bf16
    weights and stats are bitwise what zopt_muon_step gives each shape with its whole batch."""
    specs = [(4, 256, 768, torch.bfloat16, True), (3, 768, 256, torch.bfloat16, False),
             (2, 384, 1000, torch.float32, True), (1, 130, 70, torch.bfloat16, True),
             (2, 1024, 1536, torch.bfloat16, True)]
    gen = torch.Generator(device="cuda").manual_seed(5)
    sets = []
    for b, r, c, gdt, with_out in specs:
        p = torch.randn(b, r, c, generator=gen, device="cuda") * 0.02
        sets.append(dict(p=[p.clone(), p.clone()], buf=[torch.zeros_like(p), torch.zeros_like(p)],
                         out=[torch.zeros(b, r, c, dtype=torch.int16, device="cuda") if with_out else None
                              for _ in range(2)],
                         st=[zopt.new_muon_stats(b), zopt.new_muon_stats(b)], gdt=gdt, shape=(b, r, c)))
    ws = zopt.new_muon_workspace_many([(r, c, b) for b, r, c, _, _ in specs])
    for step in range(2):
        grads = [(torch.randn(*d["shape"], generator=gen, device="cuda") * 1e-3).to(d["gdt"]) for d in sets]
        zopt.muon_step_many([(d["p"][0], d["buf"][0], g, d["out"][0], d["st"][0]) for d, g in zip(sets, grads)], ws,
                            lr=8e-4)
        for d, g in zip(sets, grads):
            b, r, c = d["shape"]
            zopt.muon_step(d["p"][1], d["buf"][1], g, d["out"][1], zopt.new_muon_workspace(r, c, b), d["st"][1],
                           lr=8e-4)
        torch.cuda.synchronize()
        for d in sets:
            assert torch.equal(d["p"][0].view(torch.int32), d["p"][1].view(torch.int32)), d["shape"]
            assert torch.equal(d["buf"][0], d["buf"][1])
            if d["out"][0] is not None:
                assert torch.equal(d["out"][0], d["out"][1])
            assert torch.equal(d["st"][0], d["st"][1])


def test_many_shapes_beyond_one_elementwise_launch(zopt):
    """Ten shapes: more than one element-wise launch's worth of items (eight to a launch), so the
    momentum, statistics and update passes each run twice; every shape is bitwise its single call."""
    specs = [(1 + j % 2, 64 + 32 * j, 160 - 8 * j, torch.bfloat16 if j % 3 else torch.float32) for j in range(10)]
    gen = torch.Generator(device="cuda").manual_seed(17)
    sets = []
    for b, r, c, gdt in specs:
        p = torch.randn(b, r, c, generator=gen, device="cuda") * 0.02
        sets.append(dict(p=[p.clone(), p.clone()], buf=[torch.zeros_like(p), torch.zeros_like(p)],
                         out=[torch.zeros(b, r, c, dtype=torch.int16, device="cuda") for _ in range(2)],
                         st=[zopt.new_muon_stats(b), zopt.new_muon_stats(b)], gdt=gdt, shape=(b, r, c)))
    ws = zopt.new_muon_workspace_many([(r, c, b) for b, r, c, _ in specs])
    for step in range(2):
        grads = [(torch.randn(*d["shape"], generator=gen, device="cuda") * 1e-3).to(d["gdt"]) for d in sets]
        zopt.muon_step_many([(d["p"][0], d["buf"][0], g, d["out"][0], d["st"][0]) for d, g in zip(sets, grads)], ws,
                            lr=8e-4)
        for d, g in zip(sets, grads):
            b, r, c = d["shape"]
            zopt.muon_step(d["p"][1], d["buf"][1], g, d["out"][1], zopt.new_muon_workspace(r, c, b), d["st"][1],
                           lr=8e-4)
        torch.cuda.synchronize()
        for d in sets:
            assert torch.equal(d["p"][0].view(torch.int32), d["p"][1].view(torch.int32)), d["shape"]
            assert torch.equal(d["buf"][0], d["buf"][1]) and torch.equal(d["out"][0], d["out"][1])
            assert torch.equal(d["st"][0], d["st"][1])


@pytest.mark.parametrize("rows,cols,batch,shift", [(129, 77, 1, 1), (96, 100, 2, 2), (1, 3, 1, 0)])
def test_odd_sizes_and_unaligned_out(zopt, rows, cols, batch, shift):
    """The statistics and update kernels move 4-element vectors and finish a matrix whose size is
    not a multiple of 4 element by element; the bf16 round-out takes 8-byte stores only when the
    output allows them (a base shifted by `shift` elements does not). Master, momentum and bf16
    weights as the oracle gives them (the update within the Newton-Schulz tolerance)."""
    h = OM.MuonHyper(lr=8e-4, match_rms_adamw=True)
    gen = torch.Generator(device="cuda").manual_seed(rows * cols + shift)
    p = torch.randn(batch, rows, cols, generator=gen, device="cuda") * 0.02
    buf = torch.zeros_like(p)
    flat = torch.zeros(batch * rows * cols + shift, dtype=torch.int16, device="cuda")
    out = flat[shift:].view(batch, rows, cols)
    stats = zopt.new_muon_stats(batch)
    g = (torch.randn(batch, rows, cols, generator=gen, device="cuda") * 1e-3).bfloat16()
    p_old = p.cpu().numpy()
    zopt.muon_step(p, buf, g, out, zopt.new_muon_workspace(rows, cols), stats, lr=h.lr, match_rms_adamw=True)
    torch.cuda.synchronize()
    pn = p.cpu().numpy()
    decay = np.float32(1.0 - h.lr * h.weight_decay)
    step = np.float32(h.lr * OM.lr_scale(rows, cols, True))
    st = zopt.read_muon_stats(stats)
    for b in range(batch):
        u = OM.momentum_f32(np.zeros((rows, cols), np.float32), g[b].float().cpu().numpy(), h)
        U_ref = newton_schulz(u.astype(np.float64), steps=5)
        applied = (p_old[b] * decay - pn[b]).astype(np.float64) / float(step)
        assert rel(applied, U_ref) <= 2e-2, b
        assert not st[b]["rejected"]
    assert np.array_equal(out.cpu().numpy().view(np.uint16), f32_to_bf16_bits(pn))
    assert int(flat[:shift].abs().sum()) == 0  # nothing written before the output


def test_nan_gradient_is_rejected(zopt):
    """A NaN in the gradient reaches U through Newton-Schulz: max |U| is NaN, which the guard
    (max |U| <= guard) rejects, so the master and its bf16 weights stay as they were while the
    momentum buffer still advances (the NaN lands in it)."""
    rows, cols = 256, 512
    p = torch.randn(rows, cols, device="cuda") * 0.02
    p0 = p.clone()
    buf = torch.zeros_like(p)
    g = (torch.randn(rows, cols, device="cuda") * 1e-3).bfloat16()
    g[3, 4] = float("nan")
    out = torch.zeros(rows, cols, dtype=torch.int16, device="cuda")
    stats = zopt.new_muon_stats()
    zopt.muon_step(p, buf, g, out, zopt.new_muon_workspace(rows, cols), stats, lr=1e-3)
    torch.cuda.synchronize()
    st = zopt.read_muon_stats(stats)[0]
    assert st["rejected"] and math.isnan(st["max_abs"])
    assert torch.equal(p.view(torch.int32), p0.view(torch.int32))
    assert np.array_equal(out.cpu().numpy().view(np.uint16), f32_to_bf16_bits(p0.cpu().numpy()))
    assert math.isnan(float(buf[3, 4])) and int(torch.isnan(buf).sum()) == 1


@pytest.mark.parametrize("rows,cols", [(256, 512), (1024, 2048), (2048, 1024)])
def test_zero_gradient_decays_only(zopt, rows, cols):
    """A zero gradient with a zero momentum buffer: u = 0, so Newton-Schulz gives U = 0 (X0 =
    0 / (0 + eps)), the guard passes (max |U| = 0), nsratio is 0, and the step is the decoupled
    decay alone, p * fp32(1 - lr*wd), bit for bit: on the fused path (256 x 512), on CTA pairs
    with u read in place by the first step (1024 x 2048), and for a tall matrix (2048 x 1024)."""
    h = OM.MuonHyper(lr=8e-4)
    p = torch.randn(rows, cols, device="cuda") * 0.02
    p0 = p.cpu().numpy()
    buf = torch.zeros_like(p)
    g = torch.zeros(rows, cols, device="cuda", dtype=torch.bfloat16)
    out = torch.zeros(rows, cols, dtype=torch.int16, device="cuda")
    stats = zopt.new_muon_stats()
    zopt.muon_step(p, buf, g, out, zopt.new_muon_workspace(rows, cols), stats, lr=h.lr)
    torch.cuda.synchronize()
    st = zopt.read_muon_stats(stats)[0]
    ref = OM.muon_step(p0.copy(), np.zeros((rows, cols), np.float32), np.zeros((rows, cols), np.float32), h)
    assert not ref["rejected"] and ref["max_abs"] == 0.0
    assert not st["rejected"] and st["max_abs"] == 0.0 and st["ns_ratio"] == 0.0
    expect = p0 * np.float32(1.0 - h.lr * h.weight_decay)
    assert np.array_equal(p.cpu().numpy().view(np.uint32), expect.view(np.uint32))
    assert torch.count_nonzero(buf) == 0
    assert np.array_equal(out.cpu().numpy().view(np.uint16), f32_to_bf16_bits(expect))


@pytest.mark.parametrize("nesterov,mom,wd", [(False, 0.9, 0.0), (True, 0.5, 0.05), (False, 0.0, 0.1)])
def test_momentum_variants(zopt, nesterov, mom, wd):
    """Plain momentum (u = buf), another coefficient, no or other weight decay, and mu = 0 (u = g):
    two steps, the momentum buffer bit for bit, the applied update within 2e-2 of the fp64
    Newton-Schulz of the oracle's u, the bf16 weights bit for bit the new master's."""
    rows, cols, batch = 256, 512, 2
    h = OM.MuonHyper(lr=5e-4, momentum=mom, weight_decay=wd, nesterov=nesterov)
    gen = torch.Generator(device="cuda").manual_seed(int(mom * 100) + int(nesterov))
    p = torch.randn(batch, rows, cols, generator=gen, device="cuda") * 0.02
    buf = torch.zeros_like(p)
    out = torch.zeros(batch, rows, cols, dtype=torch.int16, device="cuda")
    ws, stats = zopt.new_muon_workspace(rows, cols, batch), zopt.new_muon_stats(batch)
    ref_buf = np.zeros((batch, rows, cols), np.float32)
    decay = np.float32(1.0 - h.lr * h.weight_decay)
    step = np.float32(h.lr * OM.lr_scale(rows, cols, True))
    for s in range(2):
        g = (torch.randn(batch, rows, cols, generator=gen, device="cuda") * 1e-3).bfloat16()
        p_old = p.cpu().numpy()
        zopt.muon_step(p, buf, g, out, ws, stats, lr=h.lr, momentum_coef=mom, weight_decay=wd, nesterov=nesterov)
        torch.cuda.synchronize()
        pn = p.cpu().numpy()
        for b in range(batch):
            u = OM.momentum_f32(ref_buf[b], g[b].float().cpu().numpy(), h)
            U_ref = newton_schulz(u.astype(np.float64), steps=5)
            applied = (p_old[b] * decay - pn[b]).astype(np.float64) / float(step)
            assert rel(applied, U_ref) <= 2e-2, (s, b)
        assert np.array_equal(buf.cpu().numpy().view(np.uint32), ref_buf.view(np.uint32))
        assert np.array_equal(out.cpu().numpy().view(np.uint16), f32_to_bf16_bits(pn))


@pytest.mark.parametrize("rows,cols,batch", [(256, 768, 2), (768, 256, 1), (1024, 1536, 1), (96, 100, 1)])
@pytest.mark.parametrize("abc", [OM.DEFAULT_ABC, (1.5, -0.5, 0.0)])
@pytest.mark.parametrize("ns_steps", [1, 5])
def test_first_step_normalises_every_path(zopt, rows, cols, batch, abc, ns_steps):
    """Where a matrix is no taller than wide and its width a multiple of 8, the momentum pass
    writes u straight into Newton-Schulz's X0, unnormalised, and the first step's products
    scale by 1 / (||u|| + eps) (X X' by its square). Covered on each path that runs a first
    step: the persistent fused launch (256 x 768), the CTA-pair launches (1024 x 1536), the
    product-by-product single-CTA launches (a zero c rules out the identity MMAs), a single step
    (the first product is also the last), and the shapes that keep the preparation pass (a tall
    matrix; a width not a multiple of 8). The update within the Newton-Schulz tolerance of the
    fp64 oracle with the same coefficients."""
    h = OM.MuonHyper(lr=8e-4, match_rms_adamw=True, ns_steps=ns_steps, abc=tuple(abc))
    gen = torch.Generator(device="cuda").manual_seed(rows + 7 * cols + ns_steps)
    p = torch.randn(batch, rows, cols, generator=gen, device="cuda") * 0.02
    buf = torch.zeros_like(p)
    out = torch.zeros(batch, rows, cols, dtype=torch.int16, device="cuda")
    stats = zopt.new_muon_stats(batch)
    g = (torch.randn(batch, rows, cols, generator=gen, device="cuda") * 1e-3).bfloat16()
    p_old = p.cpu().numpy()
    zopt.muon_step(p, buf, g, out, zopt.new_muon_workspace(rows, cols, batch), stats, lr=h.lr, ns_steps=ns_steps,
                   abc=abc)
    torch.cuda.synchronize()
    pn = p.cpu().numpy()
    decay = np.float32(1.0 - h.lr * h.weight_decay)
    step = np.float32(h.lr * OM.lr_scale(rows, cols, True))
    st = zopt.read_muon_stats(stats)
    for b in range(batch):
        u = OM.momentum_f32(np.zeros((rows, cols), np.float32), g[b].float().cpu().numpy(), h)
        U_ref = newton_schulz(u.astype(np.float64), steps=ns_steps, abc=abc)
        applied = (p_old[b] * decay - pn[b]).astype(np.float64) / float(step)
        assert rel(applied, U_ref) <= 2e-2, b
        assert abs(st[b]["update_fro"] / np.linalg.norm(U_ref) - 1) <= 2e-2
        assert not st[b]["rejected"]
    assert np.array_equal(out.cpu().numpy().view(np.uint16), f32_to_bf16_bits(pn))
