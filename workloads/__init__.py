"""Seeded synthetic workloads for the rank-local ZeRO optimizer step.

This module only describes parameter sets and draws random inputs. It holds none of the
method's arithmetic (no layout, no AdamW, no norm, no Newton-Schulz), so that the CPU
oracle and the CUDA path can both be fed the very same bytes from here without sharing
any code with each other.

Parameter shapes follow the model families the source pages train:

* a tiny d=256 decoder (smoke scale),
* the GPT-2-small body of the modded-nanogpt speedrun (train_gpt.py, model section),
* a Llama-style GQA block as in bluscript_zero_ckpt.cpp (model config),
* a 2e9-parameter AdamW-only flat shard (deg/zero.py, ZeroMaster docstring: ZeRO-2),
* a Muon Newton-Schulz stress set of 4096-wide matrices.

Recipes (stated once here, used by tests and the benchmark):

* gradients: N(0, sigma=1e-3) drawn in fp32, then rounded to bf16 by torch's own
  conversion (round-to-nearest-even);
* fp32 masters: N(0, 0.02) for 2-D parameters, 1.0 for 1-D (RMSNorm scales), as the
  C++ trainer initialises them (bluscript_zero_ckpt.cpp, init_linear / gamma init);
* AdamW moments start at zero;
* Newton-Schulz inputs: entries N(0, 1) (the stress set also divides by its Frobenius norm).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

BUCKET = 1 << 25


@dataclass(frozen=True)
class Param:
    name: str
    shape: tuple
    decay: bool  # weight decay applies (2-D); 1-D scales are excluded

    @property
    def numel(self) -> int:
        n = 1
        for s in self.shape:
            n *= s
        return n


@dataclass
class Workload:
    name: str
    adamw: list = field(default_factory=list)      # list[Param]
    muon: list = field(default_factory=list)       # list[Param] (2-D only)
    world: int = 1
    rank: int = 0
    bucket: int = BUCKET
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.95
    eps: float = 1e-8
    weight_decay: float = 0.1
    max_norm: float = 1.0
    steps: int = 3
    micro_steps: int = 1
    seed: int = 0
    zero_row_frac: float = 0.0
    ns_steps: int = 5
    lr_schedule: tuple | None = None  # (max_lr, min_lr, warmup, stable, max_steps)
    muon_lr: float = 8e-4
    muon_lr_schedule: tuple | None = None  # the same curve with Muon's (peak, floor) pair

    @property
    def adamw_numel(self) -> int:
        return sum(p.numel for p in self.adamw)

    def lr_at(self, step: int) -> float:
        """Host-side learning rate for 0-based step ``step``."""
        if self.lr_schedule is None:
            return self.lr
        return wsd_lr(step, *self.lr_schedule)

    def muon_lr_at(self, step: int) -> float:
        """Host-side Muon learning rate for 0-based step ``step`` (bluscript_zero_ckpt.cpp feeds
        both optimizer groups the one WSD curve, each with its own peak and floor)."""
        if self.muon_lr_schedule is None:
            return self.muon_lr
        return wsd_lr(step, *self.muon_lr_schedule)

    def owned_muon(self) -> list:
        """Muon matrices owned by ``rank`` under round-robin whole-parameter ownership."""
        return [p for i, p in enumerate(self.muon) if i % self.world == self.rank]


def wsd_lr(step: int, max_lr: float, min_lr: float, warmup: int, stable: int, max_steps: int) -> float:
    """Warmup-stable-decay schedule of bluscript_zero_ckpt.cpp (get_lr): linear warmup,
    a constant stretch, then cosine decay to ``min_lr``. A host input to the step."""
    if step < warmup:
        return max_lr * (step + 1) / warmup
    if step < warmup + stable:
        return max_lr
    ratio = (step - (stable + warmup)) / ((max_steps - (stable + warmup)) - 1)
    ratio = min(max(ratio, 0.0), 1.0)
    coeff = 0.5 * (1.0 + math.cos(math.pi * ratio))
    return min_lr + coeff * (max_lr - min_lr)


def wsd_short_run(max_steps: int) -> tuple:
    """The trainer's shrink rule for short runs: warmup = max(1, ms/10), stable = max(1, ms/2)."""
    warmup = max(1, max_steps // 10)
    stable = max(1, max_steps // 2)
    if warmup + stable >= max_steps - 1:
        stable = max(1, max_steps - warmup - 2)
    return warmup, stable


# --------------------------------------------------------------------------- parameter sets

def _c1() -> Workload:
    d, layers = 256, 2
    muon = []
    for l in range(layers):
        muon += [Param(f"l{l}.wqkv", (d, 3 * d), True), Param(f"l{l}.wo", (d, d), True),
                 Param(f"l{l}.gate_up", (d, 6 * d), True), Param(f"l{l}.down", (3 * d, d), True)]
    adamw = [Param("embed", (4096, d), True), Param("norm", (d,), False)]
    return Workload("c1-tiny-d256", adamw=adamw, muon=muon, steps=3, seed=0)


def _c2() -> Workload:
    d, layers, vocab = 768, 12, 50304
    muon = []
    for l in range(layers):
        muon += [Param(f"h{l}.attn.qkv", (d, 3 * d), True), Param(f"h{l}.attn.proj", (d, d), True),
                 Param(f"h{l}.mlp.fc", (d, 4 * d), True), Param(f"h{l}.mlp.proj", (4 * d, d), True)]
    adamw = [Param("wte", (vocab, d), True)]
    adamw += [Param(f"scale{i}", (d,), False) for i in range(2 * layers + 1)]
    warmup, stable = wsd_short_run(10)
    return Workload("c2-gpt2-small", adamw=adamw, muon=muon, steps=10, seed=2, zero_row_frac=0.01,
                    lr=6e-4, lr_schedule=(6e-4, 6e-5, warmup, stable, 10),
                    muon_lr_schedule=(8e-4, 8e-5, warmup, stable, 10))


def _llama_layer(l: int, d: int = 2048) -> list:
    return [Param(f"l{l}.wq", (d, d), True), Param(f"l{l}.wk", (d, 512), True),
            Param(f"l{l}.wv", (d, 512), True), Param(f"l{l}.wo", (d, d), True),
            Param(f"l{l}.gate_up", (d, 11264), True), Param(f"l{l}.down", (5632, d), True)]


def _c3() -> Workload:
    d, layers, vocab = 2048, 16, 32000
    muon = []
    for l in range(layers):
        muon += _llama_layer(l, d)
    adamw = [Param("embed", (vocab, d), True)] + [Param(f"scale{i}", (d,), False) for i in range(2 * layers + 1)]
    return Workload("c3-llama-1b-w8r0", adamw=adamw, muon=muon, world=8, rank=0, steps=5, seed=3)


def c4_params(total: int = 2_000_000_000, d: int = 2048) -> list:
    """Llama-block shapes cycled (RMSNorm scales interleaved, so the decay mask has runs)
    until ``total`` elements; the last tensor is trimmed to fit."""
    out, n, l = [], 0, 0
    while n < total:
        layer = [Param(f"l{l}.attn_norm", (d,), False)] + _llama_layer(l, d)[:4] + \
                [Param(f"l{l}.mlp_norm", (d,), False)] + _llama_layer(l, d)[4:]
        for p in layer:
            if n >= total:
                break
            k = min(p.numel, total - n)
            out.append(p if k == p.numel else Param(p.name + ".trim", (k,), p.decay))
            n += k
        l += 1
    return out


def _c4() -> Workload:
    return Workload("c4-zero2-2e9-w8r0", adamw=c4_params(), world=8, rank=0, steps=5, seed=4, micro_steps=4)


def _c5() -> Workload:
    muon = []
    for i in range(16):
        muon.append(Param(f"sq{i}", (4096, 4096), True))
    for i in range(16):
        muon.append(Param(f"wide{i}", (4096, 14336), True))
    for i in range(16):
        muon.append(Param(f"tall{i}", (14336, 4096), True))
    return Workload("c5-ns-stress", muon=muon, seed=5)


WORKLOADS = {"c1": _c1, "c2": _c2, "c3": _c3, "c4": _c4, "c5": _c5}


def get(name: str) -> Workload:
    return WORKLOADS[name]()


# --------------------------------------------------------------------------- random draws

def generator(seed: int, stream: int, device="cpu") -> torch.Generator:
    """An independent torch generator per (workload seed, named stream)."""
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + stream * 7919) & 0x7FFF_FFFF_FFFF)
    return g


def normal(shape, sigma: float, seed: int, stream: int, device="cpu", dtype=torch.float32) -> torch.Tensor:
    g = generator(seed, stream, device)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if sigma != 1.0:
        x.mul_(sigma)
    return x.to(dtype)


def grad_for(p: Param, seed: int, stream: int, zero_row_frac: float = 0.0, device="cpu",
             dtype=torch.bfloat16, sigma: float = 1e-3) -> torch.Tensor:
    """A gradient shaped like ``p``: N(0, sigma) drawn in fp32, then cast to ``dtype``;
    for 2-D parameters a seeded Bernoulli(``zero_row_frac``) picks rows that are zero."""
    g = normal(p.shape, sigma, seed, stream, device)
    if zero_row_frac > 0 and len(p.shape) == 2:
        gen = generator(seed, stream + 500_000, device)
        rows = torch.rand(p.shape[0], generator=gen, device=device) < zero_row_frac
        g[rows] = 0
    return g.to(dtype)


def master_for(p: Param, seed: int, stream: int, device="cpu") -> torch.Tensor:
    """fp32 master values: N(0, 0.02) for 2-D, ones for 1-D."""
    if len(p.shape) == 1:
        return torch.ones(p.shape, dtype=torch.float32, device=device)
    return normal(p.shape, 0.02, seed, stream, device)


def flat_masters(params: list, seed: int, device="cpu") -> list:
    return [master_for(p, seed, 10_000 + i, device).reshape(-1) for i, p in enumerate(params)]


def flat_grads(params: list, seed: int, step: int, micro: int = 0, zero_row_frac: float = 0.0,
               device="cpu", dtype=torch.bfloat16) -> list:
    base = 100_000 + step * 10_000 + micro * 1_000
    return [grad_for(p, seed, base + i, zero_row_frac, device, dtype).reshape(-1)
            for i, p in enumerate(params)]


def ns_input(rows: int, cols: int, seed: int, stream: int, device="cpu", dtype=torch.bfloat16,
             frobenius_normalise: bool = False) -> torch.Tensor:
    """A Newton-Schulz input matrix with N(0,1) entries (optionally divided by its
    Frobenius norm, as the stress set is)."""
    x = normal((rows, cols), 1.0, seed, stream, device)
    if frobenius_normalise:
        x = x / torch.linalg.vector_norm(x.double()).to(torch.float32)
    return x.to(dtype)


def shard_vector(n: int, sigma: float, seed: int, stream: int, device="cpu", dtype=torch.float32) -> torch.Tensor:
    """A flat shard-sized vector of N(0, sigma) values (used where only the shard matters)."""
    return normal((n,), sigma, seed, stream, device, dtype)
