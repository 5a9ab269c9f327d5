"""Benchmark of the rank-local ZeRO optimizer step on GB300.

One step = the whole hot path over one batch of synthetic input:
  * the ZeRO-2 flat AdamW shard of a 2e9-parameter model, rank r of W=8 (S = 250,000,000):
    gradient norm / clip / found_inf (zopt_grad_norm_clip) then the fused AdamW update with
    bf16 round-out (zopt_adamw_step);
Inputs are resident in HBM and far larger than L2 (4.5 GB per step), so no L2 flush is
needed between steps.

`python bench.py [--gpus N --steps K --warmup W] [--impl reference]` prints one JSON line.
Under torchrun (N > 1) every process simulates a different rank of the W=8 job (weak
scaling: no data-path collective); rank 0 prints.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "AdamW shard step HBM GB/s (% peak); Newton-Schulz TFLOP/s (% bf16 peak)"
WORKLOAD = "zero2-flat-shard-2e9-w8: AdamW+clip over rank r of W=8 (S=250,000,000 fp32 master/m/v, fp32 grad)"
ADAMW_BYTES = 30   # per element: read p, m, v (12) + fp32 grad (4); write p, m, v (12) + bf16 (2)
NORM_BYTES = 4     # per element: read the fp32 grad
CPU_SAMPLE = 4_000_000


def peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class Clocks:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_id: str):
        self.idx = device_id
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        rows = []
        if self.path and os.path.exists(self.path):
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) == 9:
                        rows.append(parts)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower() == "active"})
        loaded = [s for s in sm if smax and s > 0.5 * max(smax)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


def smi_id(local_rank: int) -> str:
    """The nvidia-smi id of this process's GPU (honours CUDA_VISIBLE_DEVICES)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").strip()
    if vis:
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        if local_rank < len(ids):
            return ids[local_rank]
    return str(local_rank)


def cpu_oracle_run(seconds: float = 10.0) -> dict:
    """The oracle as it stands (numpy, one core) on a bounded sample of the same workload:
    norm/clip then AdamW over CPU_SAMPLE shard elements, repeated for ~`seconds`."""
    import numpy as np

    import workloads
    from oracle import adamw as OA
    from oracle import clip as OC
    from oracle.bf16 import f32_to_bf16_bits

    w = workloads.get("c4")
    h = OA.Hyper(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
    n = CPU_SAMPLE
    p = workloads.shard_vector(n, 0.02, w.seed, 1).numpy()
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    mask = np.ones(n, np.uint8)
    mask[::1000] = 0
    g = workloads.shard_vector(n, 1e-3, w.seed, 2).numpy()
    steps, t0 = 0, time.perf_counter()
    while True:
        st = OC.clip_stats(g, w.max_norm)
        OA.step_flat_f32(p, m, v, g, mask, st["clip_coef"], h, steps + 1)
        f32_to_bf16_bits(p)
        steps += 1
        el = time.perf_counter() - t0
        if el >= seconds and steps >= 2:
            break
    gbs = (ADAMW_BYTES + NORM_BYTES) * n * steps / el / 1e9
    return {"value": round(gbs, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{steps} steps of norm/clip + AdamW + bf16 round-out over {n:,} shard elements "
                      f"(numpy fp32 exact-order oracle, {el:.1f} s)"}


def run_reference(args, rank: int) -> None:
    if rank != 0:
        return
    cpu = cpu_oracle_run(seconds=max(5.0, min(25.0, 2.0 * args.steps)))
    line = {"impl": "reference", "metric": METRIC, "value": cpu["value"], "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": None, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "l2": "inputs larger than L2"},
            "cpu_baseline": cpu, "e2e": {"value": cpu["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                                         "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, rank: int, world_procs: int, local_rank: int) -> None:
    import torch

    import workloads
    from zero_sharded_optimizer_flat_gb300 import build_lib
    build_lib.build()
    import zero_sharded_optimizer_flat_gb300 as Z

    torch.cuda.set_device(local_rank)
    dist = None
    if world_procs > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    w = workloads.get("c4")
    sim_rank = rank % w.world
    lay = Z.ShardLayout([p.numel for p in w.adamw], [p.decay for p in w.adamw], w.bucket, w.world, sim_rank)
    S = lay.shard_len if args.shard_len <= 0 else min(args.shard_len, lay.shard_len)
    if S != lay.shard_len:  # a prefix of the same parameter list, as its own layout
        lay = Z.ShardLayout([S], [1], 1 << 40, 1, 0)
    table = lay.device_table()
    gen = torch.Generator(device="cuda").manual_seed(w.seed * 100 + sim_rank)
    p = torch.randn(S, device="cuda", generator=gen).mul_(0.02)
    m = torch.zeros(S, device="cuda")
    v = torch.zeros(S, device="cuda")
    g = torch.randn(S, device="cuda", generator=gen).mul_(1e-3)
    out = torch.empty(S, dtype=torch.int16, device="cuda")
    clip, state = Z.new_clip_stats(), Z.new_adam_state()
    ws = Z.new_norm_workspace(S)
    stream = torch.cuda.current_stream()
    kw = dict(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, weight_decay=w.weight_decay, clip_stats=clip,
              adam_state=state)

    n_adamw = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_adamw)]

    def step(i=None):
        Z.grad_norm_clip(g, w.max_norm, ws, clip, stream=stream)
        if i is not None:
            ev[i][0].record(stream)
        Z.adamw_step(lay, table, p, m, v, g, out, stream=stream, **kw)
        if i is not None:
            ev[i][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(smi_id(local_rank)) as clk:
        t0.record(stream)
        for i in range(args.steps):
            step(i)
        t1.record(stream)
        torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / args.steps
    adamw_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    if dist:
        tt = torch.tensor([ms, adamw_ms], device="cuda")
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        ms, adamw_ms = float(tt[0]), float(tt[1])
        dist.barrier()
    clocks = clk.summary()

    # end to end through the public API with host buffers: the step's gradient comes from
    # pinned host memory, the clip stats are read back, each step
    g_host = g.cpu().pin_memory()
    stats_host = torch.empty(Z.CLIP_STATS_BYTES, dtype=torch.uint8).pin_memory()
    for _ in range(2):
        g.copy_(g_host, non_blocking=True)
        step()
        stats_host.copy_(clip, non_blocking=True)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        g.copy_(g_host, non_blocking=True)
        step()
        stats_host.copy_(clip, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    if dist:
        tt = torch.tensor([e2e_ms], device="cuda")
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        e2e_ms = float(tt[0])

    total_bytes = (ADAMW_BYTES + NORM_BYTES) * S * world_procs
    value = total_bytes / (ms * 1e-3) / 1e9
    pk = peaks()
    achieved = ADAMW_BYTES * S / (adamw_ms * 1e-3) / 1e9
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world_procs, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "shard_len": S, "grad_dtype": "f32", "simulated_world": w.world,
                       "l2": "inputs larger than L2 (4.5 GB/step), no flush"},
            "roofline": {"kernel": "adamw_kernel", "bound": "hbm", "achieved": round(achieved, 1),
                         "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 4),
                         "traffic": None, "peak_source": pk["source"],
                         "algorithmic_bytes_per_launch": ADAMW_BYTES * S, "avg_launch_ms": round(adamw_ms, 4)},
            "clocks": clocks,
            "e2e": {"value": round(total_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                    "h2d_bytes_per_step": 4 * S, "d2h_bytes_per_step": Z.CLIP_STATS_BYTES},
            "gpu_launches": 2 * args.steps,
        }
        if world_procs == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_oracle_run(seconds=10.0)
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--shard-len", type=int, default=0,
                    help="time a shorter prefix of the shard (profiling captures); 0 = the whole shard")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank = int(os.environ.get("RANK", "0"))
    world_procs = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    run_ours(args, rank, world_procs, local_rank)


if __name__ == "__main__":
    main()
