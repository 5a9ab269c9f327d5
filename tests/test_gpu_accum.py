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


def test_full_size_zero2_micro_steps_with_inf_run(zopt):
    """The 2e9-parameter set's rank-0 shard (S = 250,000,000): 4 bf16 micro-steps summed in
    fp32 (sampled slots bit for bit, the fused sum of squares against the oracle's over the
    whole sum), then a run with +inf injected at a seeded index of micro-step 2: found_inf is
    set and the AdamW step that follows changes nothing."""
    import workloads

    w = workloads.get("c4")
    lay = zopt.ShardLayout([p.numel for p in w.adamw], [p.decay for p in w.adamw], w.bucket, w.world, w.rank)
    S = lay.shard_len
    gen = torch.Generator(device="cuda").manual_seed(44)
    parts = [(torch.randn(S, generator=gen, device="cuda") * 1e-3).bfloat16() for _ in range(4)]
    acc, st = run(zopt, parts)
    rng = np.random.default_rng(44)
    idx = np.unique(np.concatenate([rng.integers(0, S, 100_000), [0, S - 1]]))
    idx_d = torch.from_numpy(idx).cuda()
    ref = accumulate([p[idx_d].float().cpu().numpy() for p in parts])
    assert np.array_equal(acc[idx_d].cpu().numpy().view(np.uint32), ref.view(np.uint32))
    ss = OC.sumsq(acc.cpu().numpy())
    assert close(st["sumsq"], ss) and not st["found_inf"]

    bad = int(rng.integers(0, S))
    parts[1][bad] = float("inf")
    p = torch.randn(S, generator=gen, device="cuda") * 0.02
    m, v = torch.zeros(S, device="cuda"), torch.zeros(S, device="cuda")
    out = torch.zeros(S, dtype=torch.int16, device="cuda")
    p0 = p[idx_d].clone()
    clip, state = zopt.new_clip_stats(), zopt.new_adam_state()
    ws = zopt.new_norm_workspace(S)
    for k, g in enumerate(parts):
        zopt.grad_accumulate(acc, g, first=k == 0, last=k == 3, max_norm=1.0, ws=ws, stats=clip)
    zopt.adamw_step(lay, lay.device_table(), p, m, v, acc, out, lr=w.lr, clip_stats=clip, adam_state=state)
    torch.cuda.synchronize()
    st = zopt.read_clip_stats(clip)
    assert st["found_inf"] and not st["clipped"]
    assert torch.equal(p[idx_d], p0) and int(m.abs().sum()) == 0 and int(out.abs().sum()) == 0
    assert zopt.read_adam_state(state)["step"] == 0


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
