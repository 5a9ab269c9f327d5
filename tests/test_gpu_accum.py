"""GPU parity of zopt_grad_accumulate against the oracle (deg/zero.py collect /
reduce_scatter: parts summed in fp32; grad_sq_norm of the finished sum).

Bar: the fp32 sum bit for bit; the fused clip stats as zopt_grad_norm_clip's (found_inf
exact, sumsq / norm / coef within 1e-6 relative)."""
import numpy as np
import pytest
import torch

from oracle import clip as OC
from oracle.accum import accumulate

pytestmark = pytest.mark.gpu


def close(a, b, rel=1e-6):
    return float(a) == float(b) or abs(float(a) - float(b)) <= rel * abs(float(b))


def run(Z, parts, max_norm=1.0):
    n = parts[0].numel()
    acc = torch.full((n,), float("nan"), device="cuda")  # the first part must not read it
    ws, stats = Z.new_norm_workspace(n), Z.new_clip_stats()
    for k, g in enumerate(parts):
        Z.grad_accumulate(acc, g, first=k == 0, last=k == len(parts) - 1, max_norm=max_norm, ws=ws, stats=stats)
    torch.cuda.synchronize()
    return acc, Z.read_clip_stats(stats)


@pytest.mark.parametrize("n", [1, 7, 8, 9, 1000, 8 * 1027 + 3, 2_000_003])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("k", [1, 2, 4])
def test_sum_and_stats_match_oracle(zopt, n, dtype, k):
    gen = torch.Generator(device="cuda").manual_seed(n + k)
    parts = [(torch.randn(n, generator=gen, device="cuda") * 1e-3).to(dtype) for _ in range(k)]
    acc, st = run(zopt, parts)
    ref = accumulate([p.float().cpu().numpy() for p in parts])
    assert np.array_equal(acc.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    rs = OC.clip_stats(ref, 1.0)
    assert st["found_inf"] == rs["found_inf"] and st["clipped"] == rs["clipped"]
    assert close(st["sumsq"], rs["sumsq"]) and close(st["clip_coef"], rs["clip_coef"])


@pytest.mark.parametrize("bad", [float("inf"), float("nan")])
def test_inf_in_a_middle_micro_step(zopt, bad):
    n = 100_003
    parts = [torch.randn(n, device="cuda").bfloat16() * 1e-3 for _ in range(4)]
    parts[1][12345] = bad
    acc, st = run(zopt, parts)
    assert st["found_inf"] and not st["clipped"] and st["clip_coef"] == 0.0


def test_fused_stats_agree_with_separate_norm(zopt):
    n = 3_000_017
    parts = [torch.randn(n, device="cuda").bfloat16() for _ in range(3)]
    acc, st = run(zopt, parts)
    ws, stats = zopt.new_norm_workspace(n), zopt.new_clip_stats()
    zopt.grad_norm_clip(acc, 1.0, ws, stats)
    torch.cuda.synchronize()
    sep = zopt.read_clip_stats(stats)
    assert sep["found_inf"] == st["found_inf"] and sep["clipped"] == st["clipped"]
    assert close(sep["sumsq"], st["sumsq"]) and close(sep["clip_coef"], st["clip_coef"])


def test_rejects_bad_arguments(zopt):
    acc = torch.zeros(64, device="cuda")
    g = torch.zeros(64, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(zopt.ZoptError):
        zopt.grad_accumulate(acc, g, first=True, last=True, ws=None, stats=None)  # last needs ws + stats
    with pytest.raises(zopt.ZoptError):
        zopt.grad_accumulate(acc, g.half(), first=True, last=False)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("n", [5, 8 * 1027 + 3, 1_000_003])
def test_page_locked_host_micro_grads(zopt, dtype, n):
    """Micro-step gradients read straight from pinned host memory give the device path's
    sum and stats bit for bit (and the oracle's sum)."""
    gen = torch.Generator().manual_seed(n)
    parts = [(torch.randn(n, generator=gen) * 1e-3).to(dtype) for _ in range(3)]
    host = [p.pin_memory() for p in parts]
    acc_h, st_h = run(zopt, host)
    acc_d, st_d = run(zopt, [p.cuda() for p in parts])
    assert torch.equal(acc_h, acc_d) and st_h == st_d
    ref = accumulate([p.float().numpy() for p in parts])
    assert np.array_equal(acc_h.cpu().numpy(), ref)


def test_pageable_host_micro_grad_is_refused(zopt):
    acc = torch.zeros(64, device="cuda")
    with pytest.raises(zopt.ZoptError, match="pageable"):
        zopt.grad_accumulate(acc, torch.zeros(64, dtype=torch.bfloat16), first=True, last=False)


def test_full_size_zero2_five_steps_with_inf_step(zopt):
    """The 2e9-parameter set's rank-0 shard (S = 250,000,000, W = 8) through its five stated
    steps, in the launch configuration the benchmark times: each step sums four bf16 micro-step
    gradients in fp32 (zopt_grad_accumulate, the clip stats fused into the last pass) and takes
    the AdamW step with bf16 round-out (zopt_adamw_step). Step 3 carries +inf at a seeded index of
    its second micro-step: found_inf is set, the step changes nothing and the counter stays at 2,
    so steps 4 and 5 run as t = 3 and t = 4 (their bias corrections). After every step, sampled
    slots (random, first and last, around every no-decay run edge, the poisoned index) of the sum,
    master, m, v and bf16 weights are bit for bit the oracle's, computed slot by slot; the fused
    sum of squares is within 1e-6 of the oracle's over the whole sum, the coefficient within 1e-6
    of the oracle's."""
    import workloads
    from oracle import adamw as OA
    from oracle import layout as OL
    from oracle.bf16 import f32_to_bf16_bits

    w = workloads.get("c4")
    assert w.steps == 5 and w.micro_steps == 4
    numel = [p.numel for p in w.adamw]
    decay = np.array([p.decay for p in w.adamw])
    lay = zopt.ShardLayout(numel, decay, w.bucket, w.world, w.rank)
    S = lay.shard_len
    table = lay.device_table()
    gen = torch.Generator(device="cuda").manual_seed(45)
    p = torch.randn(S, device="cuda", generator=gen) * 0.02
    m, v = torch.zeros(S, device="cuda"), torch.zeros(S, device="cuda")
    acc = torch.empty(S, device="cuda")
    out = torch.empty(S, dtype=torch.int16, device="cuda")
    clip, state, ws = zopt.new_clip_stats(), zopt.new_adam_state(), zopt.new_norm_workspace(S)
    rng = np.random.default_rng(45)
    bad_step, bad_micro, bad = 2, 1, int(rng.integers(0, S))
    runs = lay.nodecay_runs()
    edges = np.concatenate([runs.reshape(-1) + d for d in (-2, -1, 0, 1)])
    idx = np.unique(np.clip(np.concatenate([rng.integers(0, S, 200_000), [0, 1, S - 2, S - 1, bad], edges]), 0, S - 1))
    idx_d = torch.from_numpy(idx).cuda()
    owner = OL.param_of_flat(numel, OL.flat_index_of_slots(numel, w.bucket, w.world, w.rank, idx))
    dec = np.where(owner >= 0, decay[np.maximum(owner, 0)], False)
    h = OA.Hyper(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
    sp = p[idx_d].cpu().numpy()
    sm, sv = np.zeros_like(sp), np.zeros_like(sp)
    t = 0
    for s in range(w.steps):
        parts = [(torch.randn(S, generator=gen, device="cuda") * 1e-3).bfloat16() for _ in range(w.micro_steps)]
        if s == bad_step:
            parts[bad_micro][bad] = float("inf")
        for k, g in enumerate(parts):
            zopt.grad_accumulate(acc, g, first=k == 0, last=k == w.micro_steps - 1, max_norm=w.max_norm, ws=ws,
                                 stats=clip)
        zopt.adamw_step(lay, table, p, m, v, acc, out, lr=h.lr, beta1=h.beta1, beta2=h.beta2, eps=h.eps,
                        weight_decay=h.weight_decay, clip_stats=clip, adam_state=state)
        torch.cuda.synchronize()
        sg = accumulate([g[idx_d].float().cpu().numpy() for g in parts])
        assert np.array_equal(acc[idx_d].cpu().numpy().view(np.uint32), sg.view(np.uint32)), s
        st = zopt.read_clip_stats(clip)
        if s == bad_step:
            assert st["found_inf"] and not st["clipped"] and st["clip_coef"] == 0.0
        else:
            ref = OC.clip_stats(acc.cpu().numpy(), w.max_norm)
            assert not st["found_inf"] and close(st["sumsq"], ref["sumsq"])
            assert close(st["clip_coef"], ref["clip_coef"]) and st["clipped"] == ref["clipped"]
            t += 1
            sc = OA.scalars_f32(h, t)
            for mask in (dec, ~dec):
                pp, mm, vv = sp[mask], sm[mask], sv[mask]
                OA.adamw_tensor_f32(pp, mm, vv, sg[mask], np.float32(st["clip_coef"]), bool(mask is dec), sc)
                sp[mask], sm[mask], sv[mask] = pp, mm, vv
        assert np.array_equal(p[idx_d].cpu().numpy().view(np.uint32), sp.view(np.uint32)), s
        assert np.array_equal(m[idx_d].cpu().numpy().view(np.uint32), sm.view(np.uint32)), s
        assert np.array_equal(v[idx_d].cpu().numpy().view(np.uint32), sv.view(np.uint32)), s
        assert np.array_equal(out[idx_d].cpu().numpy().view(np.uint16), f32_to_bf16_bits(sp)), s
        assert zopt.read_adam_state(state)["step"] == t, s
        del parts
    assert t == 4


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("n", [1, 7, 8 * 1027 + 3, 2_000_003])
@pytest.mark.parametrize("parts,host_b", [(2, False), (4, False), (4, True)])
def test_two_parts_per_pass_bitwise(zopt, dtype, n, parts, host_b):
    """zopt_grad_accumulate2 (two micro-steps in one pass) equals one zopt_grad_accumulate call per
    part bit for bit: the fp32 sum in the same order and the fused stats; the second part may
    come from pinned host memory."""
    gen = torch.Generator(device="cuda").manual_seed(n + 10 * parts)
    gs = [(torch.randn(n, generator=gen, device="cuda") * 1e-3).to(dtype) for _ in range(parts)]
    acc1, st1 = run(zopt, gs)
    acc2 = torch.full((n,), float("nan"), device="cuda")
    ws, st = zopt.new_norm_workspace(n), zopt.new_clip_stats()
    for k in range(0, parts, 2):
        b = gs[k + 1].cpu().pin_memory() if host_b else gs[k + 1]
        zopt.grad_accumulate2(acc2, gs[k], b, first=k == 0, last=k + 2 == parts, max_norm=1.0, ws=ws, stats=st)
    torch.cuda.synchronize()
    assert torch.equal(acc1.view(torch.int32), acc2.view(torch.int32))
    assert zopt.read_clip_stats(st) == st1
