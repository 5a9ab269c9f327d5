"""GPU parity of zopt_adamw_step (with zopt_grad_norm_clip feeding the coefficient) against
the oracle's per-tensor AdamW (dmuon PR #16 op order; DeepSpeed PR #9021 grad scale on load;
deg/zero.py flat == per-tensor, gather_params bf16 round-out).

The oracle steps every parameter as a whole tensor, then its own layout picks rank r's
slots. Bar: master, m, v and the bf16 weights bit for bit (the GPU's fp32 clip coefficient
is fed to the oracle, and checked against the oracle's own within 1e-6 relative); found_inf
exact; a skipped step changes nothing and does not advance the step counter.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import adamw as OA
from oracle import clip as OC
from oracle import layout as OL
from oracle.bf16 import f32_to_bf16_bits

pytestmark = pytest.mark.gpu

SMALL = [workloads.Param("w0", (300, 77), True), workloads.Param("s0", (77,), False),
         workloads.Param("w1", (129, 50), True), workloads.Param("s1", (5,), False),
         workloads.Param("w2", (1000, 3), True), workloads.Param("s2", (1,), False),
         workloads.Param("w3", (64, 64), True)]


def bits(a):
    return np.ascontiguousarray(a).view(np.uint32)


class Case:
    """Holds a parameter set, the oracle's full tensors and the GPU shard."""

    def __init__(self, Z, params, bucket, world, rank, seed, gdtype, fused=False):
        self.Z, self.params, self.bucket, self.world, self.rank = Z, params, bucket, world, rank
        self.fused = fused  # zopt_adamw_clip_step instead of zopt_grad_norm_clip + zopt_adamw_step
        self.seed, self.gdtype = seed, gdtype
        self.numel = [p.numel for p in params]
        self.decay = [p.decay for p in params]
        self.full_p = [t.numpy().astype(np.float32) for t in workloads.flat_masters(params, seed)]
        self.full_m = [np.zeros_like(p) for p in self.full_p]
        self.full_v = [np.zeros_like(p) for p in self.full_p]
        self.idx = OL.flat_index_of_slots(self.numel, bucket, world, rank,
                                          np.arange(OL.shard_len(self.numel, bucket, world)))
        self.layout = Z.ShardLayout(self.numel, self.decay, bucket, world, rank)
        self.table = self.layout.device_table()
        S = self.layout.shard_len
        self.S = S
        self.p = torch.from_numpy(self.shard(self.full_p)).cuda()
        self.m = torch.zeros(S, device="cuda")
        self.v = torch.zeros(S, device="cuda")
        self.out = torch.zeros(S, dtype=torch.int16, device="cuda")
        self.clip = Z.new_clip_stats()
        self.state = Z.new_adam_state()
        self.ws = Z.new_norm_workspace(S)
        self.cws = Z.new_adamw_clip_workspace(S)
        self.t = 0

    def shard(self, tensors):
        return OL.gather_shard(np.concatenate(tensors), self.numel, self.bucket, self.world, self.rank, self.idx)

    def step(self, step_idx, h: OA.Hyper, max_norm=1.0, poison=None, skip_on_inf=True, zero_row_frac=0.0):
        grads = workloads.flat_grads(self.params, self.seed, step_idx, zero_row_frac=zero_row_frac, dtype=self.gdtype)
        g_full = [g.float().numpy() for g in grads]
        if poison is not None:
            k, j, val = poison
            g_full[k][j] = val
        g_shard = self.shard(g_full)
        g_dev = torch.from_numpy(g_shard).cuda().to(self.gdtype)
        if self.fused:
            self.Z.adamw_clip_step(self.layout, self.table, self.p, self.m, self.v, g_dev, self.out, lr=h.lr,
                                   max_norm=max_norm, ws=self.cws, clip_stats=self.clip, adam_state=self.state,
                                   beta1=h.beta1, beta2=h.beta2, eps=h.eps, weight_decay=h.weight_decay,
                                   skip_on_inf=skip_on_inf)
        else:
            self.Z.grad_norm_clip(g_dev, max_norm, self.ws, self.clip)
            self.Z.adamw_step(self.layout, self.table, self.p, self.m, self.v, g_dev, self.out, lr=h.lr,
                              beta1=h.beta1, beta2=h.beta2, eps=h.eps, weight_decay=h.weight_decay,
                              skip_on_inf=skip_on_inf, clip_stats=self.clip, adam_state=self.state)
        torch.cuda.synchronize()
        if self.fused:
            assert int(self.cws[:256].count_nonzero()) == 0  # every call leaves the counters at zero
        st = self.Z.read_clip_stats(self.clip)
        ref = OC.clip_stats(g_shard, max_norm)
        assert st["found_inf"] == ref["found_inf"]
        assert abs(float(st["clip_coef"]) - float(ref["clip_coef"])) <= 1e-6 * max(float(ref["clip_coef"]), 1e-30)
        if not (st["found_inf"] and skip_on_inf):
            self.t += 1
            OA.step_tensors(self.full_p, self.full_m, self.full_v, g_full, self.decay, st["clip_coef"], h, self.t)
        return st

    def compare(self):
        p = self.p.cpu().numpy()
        assert np.array_equal(bits(p), bits(self.shard(self.full_p)))
        assert np.array_equal(bits(self.m.cpu().numpy()), bits(self.shard(self.full_m)))
        assert np.array_equal(bits(self.v.cpu().numpy()), bits(self.shard(self.full_v)))
        out = self.out.cpu().numpy().view(np.uint16)
        assert np.array_equal(out, f32_to_bf16_bits(self.shard(self.full_p)))
        pad = self.idx < 0
        assert np.all(p[pad] == 0)
        assert self.Z.read_adam_state(self.state) == {"step": self.t, "arrive": 0}


H = OA.Hyper(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)


@pytest.mark.parametrize("world,rank", [(1, 0), (3, 1), (8, 0), (8, 7)])
@pytest.mark.parametrize("gdtype", [torch.bfloat16, torch.float32])
def test_small_sets_bitwise(zopt, world, rank, gdtype):
    case = Case(zopt, SMALL, 4000, world, rank, seed=11, gdtype=gdtype)
    for s in range(3):
        case.step(s, H, max_norm=0.05)  # small max_norm: the clip coefficient is active
        case.compare()


ALL_2D = [workloads.Param("a", (300, 77), True), workloads.Param("b", (129, 50), True)]
ALL_1D = [workloads.Param("s0", (777,), False), workloads.Param("s1", (5,), False), workloads.Param("s2", (4096,), False)]


@pytest.mark.parametrize("params,world,rank,null_table", [(ALL_2D, 3, 2, True), (ALL_2D, 1, 0, False),
                                                          (ALL_1D, 3, 0, False), (ALL_1D, 8, 5, False)])
def test_decay_mask_extremes_bitwise(zopt, params, world, rank, null_table):
    """Every slot decayed (no no-decay runs: the run table may then be NULL) or none decayed
    (every piece of the shard one run), several ranks; bit for bit the per-tensor oracle."""
    case = Case(zopt, params, 1000, world, rank, seed=31, gdtype=torch.bfloat16)
    if null_table:
        assert case.layout.nodecay_runs().shape[0] == 0
        case.table = None
    for s in range(2):
        case.step(s, H, max_norm=0.05)
        case.compare()


def test_c1_three_steps_bitwise(zopt):
    w = workloads.get("c1")
    case = Case(zopt, w.adamw, w.bucket, 1, 0, seed=w.seed, gdtype=torch.bfloat16)
    h = OA.Hyper(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
    for s in range(w.steps):
        case.step(s, h, max_norm=w.max_norm)
        case.compare()


def test_gpt2_small_set_ten_wsd_steps_bitwise(zopt):
    """GPT-2-small AdamW set (embedding 50304x768 + 25 scales, N = 38,652,672, 2 buckets of
    2^25), 1 % zero gradient rows, W = 1, through its ten stated steps on the trainer's WSD
    schedule for a 10-step run (bluscript_zero_ckpt.cpp, get_lr and its short-run rule: warm-up
    1 step, stable 5, cosine decay over the last 4 to the floor 6e-5): master, m, v and the bf16
    weights bit for bit after every step."""
    w = workloads.get("c2")
    assert w.steps == 10
    lrs = [w.lr_at(s) for s in range(w.steps)]
    assert lrs[9] == 6e-5 and lrs[7] < lrs[6] == lrs[1] == 6e-4  # the decay phase runs
    case = Case(zopt, w.adamw, w.bucket, 1, 0, seed=w.seed, gdtype=torch.bfloat16)
    for s in range(w.steps):
        case.step(s, OA.Hyper(lrs[s], w.beta1, w.beta2, w.eps, w.weight_decay), max_norm=w.max_norm,
                  zero_row_frac=w.zero_row_frac)
        case.compare()


def test_llama_set_rank0_of_8_five_steps_bitwise(zopt):
    """Llama-style 1.1B AdamW set (embedding 32000x2048 + 33 scales), simulated rank 0 of 8,
    through its five stated steps, bit for bit after every step."""
    w = workloads.get("c3")
    assert w.steps == 5
    case = Case(zopt, w.adamw, w.bucket, w.world, w.rank, seed=w.seed, gdtype=torch.bfloat16)
    h = OA.Hyper(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
    for s in range(w.steps):
        case.step(s, h, max_norm=w.max_norm)
        case.compare()


def test_wsd_schedule_lr_changes_each_step(zopt):
    """Per-step lr (the WSD schedule of bluscript_zero_ckpt.cpp) is a host input per call."""
    params = SMALL[:4]
    case = Case(zopt, params, 1 << 12, 2, 1, seed=5, gdtype=torch.bfloat16)
    for s in range(6):
        lr = workloads.wsd_lr(s, 6e-4, 6e-5, 1, 3, 6)
        case.step(s, OA.Hyper(lr, 0.9, 0.95, 1e-8, 0.1))
        case.compare()


@pytest.mark.parametrize("bad", [float("inf"), float("nan")])
def test_inf_grad_skips_step(zopt, bad):
    case = Case(zopt, SMALL, 4000, 1, 0, seed=3, gdtype=torch.bfloat16)
    case.step(0, H)
    case.compare()
    st = case.step(1, H, poison=(2, 17, bad))
    assert st["found_inf"] and not st["clipped"] and st["clip_coef"] == 0.0
    case.compare()  # nothing changed, step counter still 1
    case.step(2, H)
    case.compare()


def test_ragged_lengths(zopt):
    for n in (1, 3, 4, 5, 2047, 2048, 2049, 4096 * 3 + 1):
        params = [workloads.Param("a", (n,), True)]
        case = Case(zopt, params, 1 << 20, 1, 0, seed=n, gdtype=torch.float32)
        case.step(0, H)
        case.step(1, H)
        case.compare()


def test_no_output_and_no_clip_stats(zopt):
    """out_bf16 = NULL skips the round-out; d_clip = NULL means coefficient 1."""
    case = Case(zopt, SMALL, 4000, 1, 0, seed=9, gdtype=torch.bfloat16)
    grads = workloads.flat_grads(SMALL, 9, 0)
    g_full = [g.float().numpy() for g in grads]
    g_dev = torch.from_numpy(case.shard(g_full)).cuda().bfloat16()
    zopt.adamw_step(case.layout, case.table, case.p, case.m, case.v, g_dev, None, lr=H.lr, clip_stats=None,
                    adam_state=case.state)
    torch.cuda.synchronize()
    OA.step_tensors(case.full_p, case.full_m, case.full_v, g_full, case.decay, 1.0, H, 1)
    assert np.array_equal(bits(case.p.cpu().numpy()), bits(case.shard(case.full_p)))
    assert int(case.out.abs().sum()) == 0


def test_full_size_zero2_shard_sampled(zopt):
    """The 2e9-parameter ZeRO-2 shard (rank 0 of 8, S = 250,000,000), in the launch
    configuration the benchmark times: sampled slots checked bit for bit against the oracle
    computed one element at a time."""
    w = workloads.get("c4")
    numel = [p.numel for p in w.adamw]
    decay = np.array([p.decay for p in w.adamw])
    lay = zopt.ShardLayout(numel, decay, w.bucket, w.world, w.rank)
    S = lay.shard_len
    table = lay.device_table()
    gen = torch.Generator(device="cuda").manual_seed(4)
    p = torch.randn(S, device="cuda", generator=gen) * 0.02
    m = torch.zeros(S, device="cuda")
    v = torch.zeros(S, device="cuda")
    out = torch.empty(S, dtype=torch.int16, device="cuda")
    clip, state = zopt.new_clip_stats(), zopt.new_adam_state()
    ws = zopt.new_norm_workspace(S)
    rng = np.random.default_rng(4)
    # samples: random slots, the first and last slots, and slots around every no-decay run edge
    runs = lay.nodecay_runs()
    edges = np.concatenate([runs.reshape(-1) + d for d in (-2, -1, 0, 1)])
    idx = np.unique(np.clip(np.concatenate([rng.integers(0, S, 200_000), [0, 1, S - 2, S - 1], edges]), 0, S - 1))
    idx_d = torch.from_numpy(idx).cuda()
    flat = OL.flat_index_of_slots(numel, w.bucket, w.world, w.rank, idx)
    owner = OL.param_of_flat(numel, flat)
    dec = np.where(owner >= 0, decay[np.maximum(owner, 0)], False)
    h = OA.Hyper(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
    sp = p[idx_d].cpu().numpy()
    sm = np.zeros_like(sp)
    sv = np.zeros_like(sp)
    for t in range(1, 3):
        g = torch.randn(S, device="cuda", generator=gen) * 1e-3
        zopt.grad_norm_clip(g, w.max_norm, ws, clip)
        zopt.adamw_step(lay, table, p, m, v, g, out, lr=h.lr, beta1=h.beta1, beta2=h.beta2, eps=h.eps,
                        weight_decay=h.weight_decay, clip_stats=clip, adam_state=state)
        torch.cuda.synchronize()
        st = zopt.read_clip_stats(clip)
        sg = g[idx_d].cpu().numpy()
        ref_ss = OC.sumsq(g.cpu().numpy())
        assert abs(st["sumsq"] - ref_ss) <= 1e-6 * ref_ss
        sc = OA.scalars_f32(h, t)
        for mask in (dec, ~dec):
            pp, mm, vv = sp[mask], sm[mask], sv[mask]
            OA.adamw_tensor_f32(pp, mm, vv, sg[mask], st["clip_coef"], bool(mask is dec), sc)
            sp[mask], sm[mask], sv[mask] = pp, mm, vv
        assert np.array_equal(bits(p[idx_d].cpu().numpy()), bits(sp))
        assert np.array_equal(bits(m[idx_d].cpu().numpy()), bits(sm))
        assert np.array_equal(bits(v[idx_d].cpu().numpy()), bits(sv))
        assert np.array_equal(out[idx_d].cpu().numpy().view(np.uint16), f32_to_bf16_bits(sp))
    assert zopt.read_adam_state(state)["step"] == 2


def test_full_size_zero2_shard_clip_step_sampled(zopt):
    """zopt_adamw_clip_step on the 2e9-parameter ZeRO-2 shard (rank 0 of 8, S = 250,000,000, an
    fp32 gradient): one cooperative wave over about 120,000 tiles, each block summing and then
    updating its own run. The sum of squares within 1e-6 of the oracle's over the whole shard;
    sampled slots (random, both ends, every no-decay run edge) bit for bit the oracle's step on
    the call's own clip coefficient; the counters back at zero after each call."""
    w = workloads.get("c4")
    numel = [p.numel for p in w.adamw]
    decay = np.array([p.decay for p in w.adamw])
    lay = zopt.ShardLayout(numel, decay, w.bucket, w.world, w.rank)
    S = lay.shard_len
    table = lay.device_table()
    gen = torch.Generator(device="cuda").manual_seed(14)
    p = torch.randn(S, device="cuda", generator=gen) * 0.02
    m = torch.zeros(S, device="cuda")
    v = torch.zeros(S, device="cuda")
    out = torch.empty(S, dtype=torch.int16, device="cuda")
    clip, state = zopt.new_clip_stats(), zopt.new_adam_state()
    cws = zopt.new_adamw_clip_workspace(S)
    rng = np.random.default_rng(14)
    runs = lay.nodecay_runs()
    edges = np.concatenate([runs.reshape(-1) + d for d in (-2, -1, 0, 1)])
    idx = np.unique(np.clip(np.concatenate([rng.integers(0, S, 200_000), [0, 1, S - 2, S - 1], edges]), 0, S - 1))
    idx_d = torch.from_numpy(idx).cuda()
    flat = OL.flat_index_of_slots(numel, w.bucket, w.world, w.rank, idx)
    owner = OL.param_of_flat(numel, flat)
    dec = np.where(owner >= 0, decay[np.maximum(owner, 0)], False)
    h = OA.Hyper(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
    sp = p[idx_d].cpu().numpy()
    sm = np.zeros_like(sp)
    sv = np.zeros_like(sp)
    for t in range(1, 3):
        g = torch.randn(S, device="cuda", generator=gen) * 1e-3
        zopt.adamw_clip_step(lay, table, p, m, v, g, out, lr=h.lr, max_norm=w.max_norm, ws=cws, clip_stats=clip,
                             adam_state=state, beta1=h.beta1, beta2=h.beta2, eps=h.eps, weight_decay=h.weight_decay)
        torch.cuda.synchronize()
        st = zopt.read_clip_stats(clip)
        ref_ss = OC.sumsq(g.cpu().numpy())
        assert abs(st["sumsq"] - ref_ss) <= 1e-6 * ref_ss
        assert st["clipped"] == 1 and 0.0 < st["clip_coef"] < 1.0  # norm ~16 against max_norm 1
        assert cws[:256].count_nonzero() == 0
        sg = g[idx_d].cpu().numpy()
        sc = OA.scalars_f32(h, t)
        for mask in (dec, ~dec):
            pp, mm, vv = sp[mask], sm[mask], sv[mask]
            OA.adamw_tensor_f32(pp, mm, vv, sg[mask], st["clip_coef"], bool(mask is dec), sc)
            sp[mask], sm[mask], sv[mask] = pp, mm, vv
        assert np.array_equal(bits(p[idx_d].cpu().numpy()), bits(sp))
        assert np.array_equal(bits(m[idx_d].cpu().numpy()), bits(sm))
        assert np.array_equal(bits(v[idx_d].cpu().numpy()), bits(sv))
        assert np.array_equal(out[idx_d].cpu().numpy().view(np.uint16), f32_to_bf16_bits(sp))
    assert zopt.read_adam_state(state)["step"] == 2


H_BETA1_ZERO = OA.Hyper(lr=1e-3, beta1=0.0, beta2=0.99, eps=1e-8, weight_decay=0.1)


@pytest.mark.parametrize("gdtype,h", [(torch.bfloat16, H), (torch.float32, H), (torch.bfloat16, H_BETA1_ZERO)])
def test_rescale_step_bitwise_and_close_to_direct(zopt, gdtype, h):
    """zopt_adamw_rescale_step (DeepSpeed PR #9021 adam_rescale_step): bit for bit the oracle's
    re-targeting; a rescale to the same scale changes nothing; the result is the step taken
    directly on the new scale up to rounding (the page measures 7.5e-6 of the update). Also with
    betas (0, 0.99), the case the page's rollback (a division by the betas) could not undo."""
    case = Case(zopt, SMALL, 4000, 3, 1, seed=21, gdtype=gdtype)
    for s in range(2):
        case.step(s, h, max_norm=1e9)  # warm moments, coefficient 1
    grads = workloads.flat_grads(SMALL, 21, 2, dtype=gdtype)
    g = case.shard([x.float().numpy() for x in grads])
    g_dev = torch.from_numpy(g).cuda().to(gdtype)
    before = [t.clone() for t in (case.p, case.m, case.v)]
    kw = dict(lr=h.lr, beta1=h.beta1, beta2=h.beta2, eps=h.eps, weight_decay=h.weight_decay)
    zopt.adamw_step(case.layout, case.table, case.p, case.m, case.v, g_dev, case.out, clip_stats=None,
                    adam_state=case.state, **kw)  # speculative step t = 3 on the unscaled gradient
    spec = [t.clone() for t in (case.p, case.m, case.v)]
    zopt.adamw_rescale_step(case.layout, case.p, case.m, case.v, g_dev, case.out, old_scale=1.0, new_scale=1.0,
                            adam_state=case.state, **kw)
    torch.cuda.synchronize()
    for a, b in zip(spec, (case.p, case.m, case.v)):
        assert torch.equal(a, b)
    zopt.adamw_rescale_step(case.layout, case.p, case.m, case.v, g_dev, case.out, old_scale=1.0, new_scale=0.37,
                            adam_state=case.state, **kw)
    torch.cuda.synchronize()
    ref = [t.cpu().numpy() for t in spec]
    OA.rescale_step_f32(*ref, g, 1.0, 0.37, h, 3)
    for r, t in zip(ref, (case.p, case.m, case.v)):
        assert np.array_equal(r.view(np.uint32), t.cpu().numpy().view(np.uint32))
    assert np.array_equal(case.out.cpu().numpy().view(np.uint16), f32_to_bf16_bits(ref[0]))
    # against the step taken directly on the new scale
    direct = [t.cpu().numpy() for t in before]
    mask = OL.decay_mask_of_shard(case.decay, case.numel, case.bucket, case.world, case.rank)
    OA.step_flat_f32(*direct, g, mask, np.float32(0.37), h, 3)
    upd = np.max(np.abs(direct[0] - before[0].cpu().numpy()))
    # 1e-4 of the update, plus the two roundings of weights near 1 (the RMSNorm scales)
    assert np.all(np.abs(direct[0] - ref[0]) <= 1e-4 * upd + 2 * np.spacing(np.abs(direct[0])))
    assert zopt.read_adam_state(case.state)["step"] == 3


def test_rescale_to_the_clip_coefficient(zopt):
    case = Case(zopt, SMALL, 4000, 1, 0, seed=22, gdtype=torch.bfloat16)
    case.step(0, H, max_norm=1e9)
    grads = workloads.flat_grads(SMALL, 22, 1)
    g = case.shard([x.float().numpy() for x in grads])
    g_dev = torch.from_numpy(g).cuda().bfloat16()
    zopt.adamw_step(case.layout, case.table, case.p, case.m, case.v, g_dev, case.out, lr=H.lr, clip_stats=None,
                    adam_state=case.state)
    spec = [t.cpu().numpy() for t in (case.p, case.m, case.v)]
    zopt.grad_norm_clip(g_dev, 0.01, case.ws, case.clip)  # the final clip, computed afterwards
    zopt.adamw_rescale_step(case.layout, case.p, case.m, case.v, g_dev, None, lr=H.lr, old_scale=1.0,
                            clip_stats=case.clip, adam_state=case.state)
    torch.cuda.synchronize()
    coef = zopt.read_clip_stats(case.clip)["clip_coef"]
    assert coef < 1
    OA.rescale_step_f32(*spec, g, 1.0, float(coef), H, 2)
    for r, t in zip(spec, (case.p, case.m, case.v)):
        assert np.array_equal(r.view(np.uint32), t.cpu().numpy().view(np.uint32))


@pytest.mark.parametrize("n", [1, 7, 2047, 2048, 2049, 6149])
def test_rescale_tile_edges(zopt, n):
    """The rescale kernel walks whole 2048-element tiles and then the tail element by element:
    shards below one tile, exactly one or two tiles, and a tile plus a ragged tail are each bit
    for bit the oracle's re-targeting, bf16 weights included."""
    case = Case(zopt, [workloads.Param("w", (n,), True)], 1 << 20, 1, 0, seed=n, gdtype=torch.bfloat16)
    for s in range(2):
        case.step(s, H, max_norm=1e9)
    g = case.shard([x.float().numpy() for x in workloads.flat_grads(case.params, n, 2, dtype=torch.bfloat16)])
    g_dev = torch.from_numpy(g).cuda().bfloat16()
    zopt.adamw_step(case.layout, case.table, case.p, case.m, case.v, g_dev, case.out, lr=H.lr, clip_stats=None,
                    adam_state=case.state)
    spec = [t.cpu().numpy() for t in (case.p, case.m, case.v)]
    zopt.adamw_rescale_step(case.layout, case.p, case.m, case.v, g_dev, case.out, lr=H.lr, old_scale=1.0,
                            new_scale=0.5, adam_state=case.state)
    torch.cuda.synchronize()
    OA.rescale_step_f32(*spec, g, 1.0, 0.5, H, 3)
    for r, t in zip(spec, (case.p, case.m, case.v)):
        assert np.array_equal(r.view(np.uint32), t.cpu().numpy().view(np.uint32))
    assert np.array_equal(case.out.cpu().numpy().view(np.uint16), f32_to_bf16_bits(spec[0]))


@pytest.mark.parametrize("gdtype", [torch.bfloat16, torch.float32])
def test_rescale_many_tiles_per_block(zopt, gdtype):
    """A shard of several 2048-element tiles per block (9,000,001 elements: over 4,000 whole
    tiles for a grid of at most a few hundred blocks) and a ragged tail: the kernel's loop that
    issues a half of its next tile's loads while it computes the rest of this one is bit for bit
    the oracle's re-targeting on every element, bf16 weights included."""
    n = 9_000_001
    rng = np.random.default_rng(17)
    p = rng.normal(0.0, 0.02, n).astype(np.float32)
    m = rng.normal(0.0, 1e-3, n).astype(np.float32)
    v = np.abs(rng.normal(0.0, 1e-5, n)).astype(np.float32)
    g_dev = torch.from_numpy(rng.normal(0.0, 1e-2, n).astype(np.float32)).cuda().to(gdtype)
    g = g_dev.float().cpu().numpy()
    lay = zopt.ShardLayout([n], [1], 1 << 24, 1, 0)
    assert lay.shard_len == n
    dp, dm, dv = (torch.from_numpy(a.copy()).cuda() for a in (p, m, v))
    out = torch.empty(n, dtype=torch.int16, device="cuda")
    state = zopt.new_adam_state()
    state.view(torch.int64)[0] = 3  # the step being re-targeted is t = 3
    zopt.adamw_rescale_step(lay, dp, dm, dv, g_dev, out, lr=H.lr, old_scale=1.0, new_scale=0.37, adam_state=state)
    torch.cuda.synchronize()
    OA.rescale_step_f32(p, m, v, g, 1.0, 0.37, H, 3)
    for r, t in zip((p, m, v), (dp, dm, dv)):
        assert np.array_equal(bits(r), bits(t.cpu().numpy()))
    assert np.array_equal(out.cpu().numpy().view(np.uint16), f32_to_bf16_bits(p))


def test_rescale_division_by_constant_is_exact(zopt):
    """The rescale kernel forms sqrt(v) / c, c = sqrt(1 - beta2^t), with a reciprocal and one FMA
    correction (Markstein's method) instead of an IEEE division. For every bit pattern of
    v >= 0 (and the positive NaNs) the result equals __fdiv_rn's, at each c of a grid of betas
    and steps and at 200 random c in (0, 1]."""
    cs = {1.0, float(np.float32(2.0 ** -20))}
    for b2 in (0.9, 0.95, 0.98, 0.99, 0.995, 0.999, 0.9999, 0.99999):
        for t in (1, 2, 3, 5, 7, 10, 30, 100, 300, 1000, 3000, 10000, 100000, 1000000):
            cs.add(float(np.float32(np.sqrt(1.0 - b2 ** t))))
    rng = np.random.default_rng(7)
    cs.update(float(x) for x in rng.uniform(2.0 ** -20, 1.0, 200).astype(np.float32))
    counter = torch.zeros(1, dtype=torch.int64, device="cuda")
    for c in sorted(cs):
        assert 0.0 < c <= 1.0
        zopt.selftest_div_by_const(c, counter)
    torch.cuda.synchronize()
    assert int(counter.item()) == 0


def test_rescale_division_selftest_rejects_bad_arguments(zopt):
    counter = torch.zeros(1, dtype=torch.int64, device="cuda")
    for c in (0.0, -1.0, 1.5, float("nan")):
        with pytest.raises(zopt.ZoptError):
            zopt.selftest_div_by_const(c, counter)


@pytest.mark.parametrize("hp", [OA.Hyper(lr=3e-4, beta1=0.0, beta2=0.999, eps=1e-8, weight_decay=0.0),
                                OA.Hyper(lr=1e-2, beta1=0.9, beta2=0.999, eps=1e-6, weight_decay=0.01),
                                OA.Hyper(lr=0.0, beta1=0.8, beta2=0.9, eps=1e-8, weight_decay=0.1),
                                OA.Hyper(lr=1e-3, beta1=0.99, beta2=0.9999, eps=1e-10, weight_decay=1.0)])
def test_other_hyperparameters_bitwise(zopt, hp):
    """The exact-order step holds for any hyper-parameters: no momentum (beta1 = 0), a slow second
    moment (beta2 = 0.999 / 0.9999: a small bias-correction constant), lr = 0 (decay only by
    1 - 0 = 1: the master stays put), no weight decay, a large decay; four steps each, master,
    m, v and bf16 weights bit for bit the oracle's."""
    case = Case(zopt, SMALL, 4000, 2, 1, seed=31, gdtype=torch.bfloat16)
    for s in range(4):
        case.step(s, hp, max_norm=1.0)
        case.compare()


# --------------------------------------------------------------------------- zopt_adamw_clip_step
# The norm / clip reduction and the step in one launch. Same bar as the two-call path: the
# GPU's own clip coefficient (read back) drives the oracle's per-tensor AdamW, master, m, v and
# the bf16 weights bit for bit; the coefficient within 1e-6 of the oracle's; found_inf exact; a
# skipped step changes nothing; and every call leaves the workspace's counters at zero.


@pytest.mark.parametrize("world,rank", [(1, 0), (3, 1), (8, 7)])
@pytest.mark.parametrize("gdtype", [torch.bfloat16, torch.float32])
def test_clip_step_small_sets_bitwise(zopt, world, rank, gdtype):
    case = Case(zopt, SMALL, 4000, world, rank, seed=11, gdtype=gdtype, fused=True)
    for s in range(3):
        case.step(s, H, max_norm=0.05)  # the clip coefficient is active
        case.compare()


@pytest.mark.parametrize("bad", [float("inf"), float("nan")])
def test_clip_step_nonfinite_grad_skips_inside_a_sequence(zopt, bad):
    case = Case(zopt, SMALL, 4000, 1, 0, seed=3, gdtype=torch.bfloat16, fused=True)
    case.step(0, H)
    case.compare()
    st = case.step(1, H, poison=(2, 17, bad))
    assert st["found_inf"] and not st["clipped"] and st["clip_coef"] == 0.0
    case.compare()  # nothing changed, step counter still 1
    case.step(2, H)
    case.step(3, H, max_norm=1e30)  # no clipping: coefficient 1
    case.compare()


def test_clip_step_ragged_lengths(zopt):
    """Shards shorter than a tile, a tile and a vector off it, several tiles and a tail: the
    blocks' runs, the 8-element sums of squares and the scalar tail all meet the oracle."""
    for n in (1, 3, 7, 8, 9, 2047, 2048, 2049, 4096 * 3 + 1, 999_999):
        params = [workloads.Param("a", (n,), True)]
        case = Case(zopt, params, 1 << 20, 1, 0, seed=n, gdtype=torch.float32, fused=True)
        case.step(0, H, max_norm=0.5)
        case.step(1, H, max_norm=0.5)
        case.compare()


@pytest.mark.parametrize("name", ["c2", "c3"])
def test_clip_step_parameter_sets_bitwise(zopt, name):
    """The GPT-2-small set (W = 1, 38.65 M slots) and the 1.1B set's rank 0 of 8 (8.2 M), through
    their stated steps (the GPT-2-small set on its WSD schedule), bit for bit after every step."""
    w = workloads.get(name)
    case = Case(zopt, w.adamw, w.bucket, w.world, w.rank, seed=w.seed, gdtype=torch.bfloat16, fused=True)
    for s in range(w.steps):
        case.step(s, OA.Hyper(w.lr_at(s), w.beta1, w.beta2, w.eps, w.weight_decay), max_norm=w.max_norm,
                  zero_row_frac=w.zero_row_frac)
        case.compare()


def test_clip_step_in_a_cuda_graph(zopt):
    """Captured once and replayed, the fused call gives what the same calls eagerly give: the
    stats, the weights and the step counter stay on the device, the workspace's counters return
    to zero."""
    cases = [Case(zopt, SMALL, 4000, 2, 1, seed=21, gdtype=torch.bfloat16, fused=True) for _ in range(2)]
    g = [torch.from_numpy(cases[0].shard([x.float().numpy() for x in workloads.flat_grads(SMALL, 21, s)])).cuda()
         .bfloat16() for s in range(3)]
    g_in = g[0].clone()

    def call(c, grad):
        zopt.adamw_clip_step(c.layout, c.table, c.p, c.m, c.v, grad, c.out, lr=H.lr, max_norm=0.05, ws=c.cws,
                             clip_stats=c.clip, adam_state=c.state)

    eager, graphed = cases
    call(graphed, g_in)  # the first call sets up the launch outside the capture
    call(eager, g[0])
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            call(graphed, g_in)
    for s in (1, 2):
        g_in.copy_(g[s])
        graph.replay()
        call(eager, g[s])
    torch.cuda.synchronize()
    for a, b in ((graphed.p, eager.p), (graphed.m, eager.m), (graphed.v, eager.v), (graphed.out, eager.out)):
        assert torch.equal(a, b)
    assert torch.equal(graphed.clip, eager.clip)
    assert zopt.read_adam_state(graphed.state) == zopt.read_adam_state(eager.state) == {"step": 3, "arrive": 0}
    assert int(graphed.cws[:256].count_nonzero()) == 0
