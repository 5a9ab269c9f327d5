"""A whole optimizer step captured once in a CUDA graph and replayed.

Every entry point is asynchronous on the caller's stream, never synchronises the host and
allocates no device memory, and every per-step quantity (clip coefficient, found_inf, the
AdamW step counter and its bias corrections, the Newton-Schulz norms, the Muon guard) lives on
the device. So the step can be captured once and replayed: each replay must leave bit for bit
the state that the same calls leave when issued one by one, and the device-side step counter
must advance once per replay.
"""
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

PARAMS = [workloads.Param("w0", (300, 77), True), workloads.Param("s0", (77,), False),
          workloads.Param("w1", (1024, 1000), True), workloads.Param("s1", (5,), False)]
NS_SHAPES = [(2, 256, 768), (1, 1024, 1100)]
MUON_SHAPE = (2, 128, 256)


class Arm:
    """One copy of the optimizer state and its workspaces."""

    def __init__(self, Z, init):
        self.Z = Z
        numel = [p.numel for p in PARAMS]
        self.lay = Z.ShardLayout(numel, [p.decay for p in PARAMS], 1 << 20, 1, 0)
        self.table = self.lay.device_table()
        S = self.lay.shard_len
        self.g = torch.zeros(S, device="cuda")
        self.p = init["p"].clone()
        self.m = torch.zeros(S, device="cuda")
        self.v = torch.zeros(S, device="cuda")
        self.out = torch.zeros(S, dtype=torch.int16, device="cuda")
        self.clip = Z.new_clip_stats()
        self.state = Z.new_adam_state()
        self.nws = Z.new_norm_workspace(S)
        self.X = [torch.zeros(b, r, c, dtype=torch.bfloat16, device="cuda") for b, r, c in NS_SHAPES]
        self.nsws = Z.new_ns_workspace_many([(r, c, b) for b, r, c in NS_SHAPES])
        b, r, c = MUON_SHAPE
        self.mp = init["mp"].clone()
        self.mbuf = torch.zeros(b, r, c, device="cuda")
        self.mout = torch.zeros(b, r, c, dtype=torch.int16, device="cuda")
        self.mst = Z.new_muon_stats(b)
        self.mws = Z.new_muon_workspace_many([(r, c, b)])

    def step(self, inp):
        Z = self.Z
        Z.grad_accumulate(self.g, inp["micro"][0], first=True, last=False)
        Z.grad_accumulate(self.g, inp["micro"][1], first=False, last=True, max_norm=1.0, ws=self.nws, stats=self.clip)
        Z.adamw_step(self.lay, self.table, self.p, self.m, self.v, self.g, self.out, lr=1e-3, clip_stats=self.clip,
                     adam_state=self.state)
        Z.ns_orthogonalize_many(list(zip(inp["G"], self.X)), self.nsws, steps=5)
        Z.muon_step_many([(self.mp, self.mbuf, inp["mg"], self.mout, self.mst)], self.mws, lr=8e-4)

    def tensors(self):
        return [self.g, self.p, self.m, self.v, self.out, self.clip, self.state, *self.X, self.mp, self.mbuf,
                self.mout, self.mst]


def test_whole_step_replayed_from_a_cuda_graph(zopt):
    gen = torch.Generator(device="cuda").manual_seed(23)
    S = zopt.ShardLayout([p.numel for p in PARAMS], None, 1 << 20, 1, 0).shard_len
    init = {"p": torch.randn(S, generator=gen, device="cuda") * 0.02,
            "mp": torch.randn(*MUON_SHAPE, generator=gen, device="cuda") * 0.02}
    inp = {"micro": [(torch.randn(S, generator=gen, device="cuda") * 1e-3).to(torch.bfloat16) for _ in range(2)],
           "G": [torch.randn(b, r, c, generator=gen, device="cuda").to(torch.bfloat16) for b, r, c in NS_SHAPES],
           "mg": (torch.randn(*MUON_SHAPE, generator=gen, device="cuda") * 1e-3).to(torch.bfloat16)}
    Arm(zopt, init).step(inp)  # first use of every entry point (one-time setup) outside the capture
    torch.cuda.synchronize()

    eager, graphed = Arm(zopt, init), Arm(zopt, init)
    for _ in range(3):
        eager.step(inp)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        graphed.step(inp)
    torch.cuda.synchronize()
    # capturing issues no work: the graphed state is still the initial one
    assert zopt.read_adam_state(graphed.state)["step"] == 0
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert zopt.read_adam_state(eager.state)["step"] == 3
    for k, (a, b) in enumerate(zip(eager.tensors(), graphed.tensors())):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), k
    assert zopt.take_device_error() == 0


def test_replayed_accumulation_reads_the_pinned_buffer_anew(zopt):
    """The accumulation of micro-step gradients held in pinned host memory, captured once: the
    graph keeps the buffers' addresses, so each replay sums what the host wrote there since,
    bit for bit what the eager calls give for the same contents."""
    n = 1_000_003
    gen = torch.Generator().manual_seed(7)
    host = [torch.empty(n, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    acc_g, acc_e = torch.empty(n, device="cuda"), torch.empty(n, device="cuda")
    ws_g, ws_e = zopt.new_norm_workspace(n), zopt.new_norm_workspace(n)
    st_g, st_e = zopt.new_clip_stats(), zopt.new_clip_stats()

    def step(acc, ws, st):
        zopt.grad_accumulate(acc, host[0], first=True, last=False)
        zopt.grad_accumulate(acc, host[1], first=False, last=True, max_norm=1.0, ws=ws, stats=st)

    for h in host:
        h.copy_(torch.randn(n, generator=gen).to(torch.bfloat16))
    step(acc_e, ws_e, st_e)  # first use outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(acc_g, ws_g, st_g)
    torch.cuda.synchronize()
    for rnd in range(3):
        for h in host:  # new contents, same addresses
            h.copy_((torch.randn(n, generator=gen) * (rnd + 1)).to(torch.bfloat16))
        g.replay()
        step(acc_e, ws_e, st_e)
        torch.cuda.synchronize()
        assert torch.equal(acc_g.view(torch.int32), acc_e.view(torch.int32)), rnd
        assert torch.equal(st_g, st_e), rnd
        want = host[0].float() + host[1].float()
        assert torch.equal(acc_g.cpu(), want), rnd


def test_replayed_two_part_accumulation(zopt):
    """zopt_grad_accumulate2 captured once (one part on the device, one in pinned host memory):
    every replay equals the eager calls bit for bit, sum and stats."""
    n = 777_777
    gen = torch.Generator().manual_seed(9)
    dev = [(torch.randn(n, generator=gen) * 1e-3).to(torch.bfloat16).cuda() for _ in range(2)]
    host = [torch.empty(n, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    out = {}
    for arm in ("graph", "eager"):
        out[arm] = (torch.empty(n, device="cuda"), zopt.new_norm_workspace(n), zopt.new_clip_stats())

    def step(acc, ws, st):
        zopt.grad_accumulate2(acc, dev[0], host[0], first=True, last=False)
        zopt.grad_accumulate2(acc, dev[1], host[1], first=False, last=True, max_norm=1.0, ws=ws, stats=st)

    for h in host:
        h.copy_((torch.randn(n, generator=gen) * 1e-3).to(torch.bfloat16))
    step(*out["eager"])  # first use outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(*out["graph"])
    torch.cuda.synchronize()
    for rnd in range(2):
        for h in host:
            h.copy_((torch.randn(n, generator=gen) * 1e-3).to(torch.bfloat16))
        g.replay()
        step(*out["eager"])
        torch.cuda.synchronize()
        assert torch.equal(out["graph"][0].view(torch.int32), out["eager"][0].view(torch.int32)), rnd
        assert torch.equal(out["graph"][2], out["eager"][2]), rnd
