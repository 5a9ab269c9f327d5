"""Benchmark of the rank-local ZeRO optimizer step on GB300.

One step = the whole hot path over one batch of synthetic input:
  * the ZeRO-2 flat AdamW shard of a 2e9-parameter model, rank r of W=8 (S = 250,000,000):
    4 bf16 micro-step gradients summed into the fp32 shard gradient, the last pass also
    producing the norm / clip / found_inf stats (zopt_grad_accumulate), then the fused AdamW
    update with bf16 round-out (zopt_adamw_step);
  * Muon's Newton-Schulz (5 steps, bf16) on the stress set of 48 whole matrices: 16 each of
    4096x4096, 4096x14336 and 14336x4096 (zopt_ns_orthogonalize_many, one call over the shapes).
Inputs are resident in HBM and far larger than L2 (~13 GB touched per step), so no L2 flush
is needed between steps. `value` is the AdamW part's HBM throughput (66 algorithmic bytes per
shard element: 36 for the accumulation, 30 for the update, / the part's time); `ns.value` the
Newton-Schulz TFLOP/s (algorithmic flops, symmetric halves counted once).

`python bench.py [--gpus N --steps K --warmup W] [--impl reference]` prints one JSON line.
Under torchrun (N > 1) every process simulates a different rank of the W=8 job and runs its
own copy of the Newton-Schulz set (weak scaling: no data-path collective); rank 0 prints.
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
WORKLOAD = ("zero2-flat-shard-2e9-w8 + ns-stress-48: rank r of W=8 (S=250,000,000): 4 bf16 micro-step grads "
            "summed into fp32 with the clip stats fused into the last pass, then AdamW with bf16 round-out; "
            "Newton-Schulz (5 steps, bf16) on 16 x 4096^2, 16 x 4096x14336, 16 x 14336x4096")
ADAMW_BYTES = 30   # per element: read p, m, v (12) + fp32 grad (4); write p, m, v (12) + bf16 (2)
# DRAM bytes per element of one adamw_kernel launch from an ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum on a 64 Mi-element shard prefix, 1.9 GB per launch, scaled by the element
# count), valid while the kernel's sources hash to ADAMW_SRC_DIGEST (otherwise the traffic is
# reported as null)
ADAMW_TRAFFIC_PER_ELEM = (1073795712 + 881538688) / 67108864
ADAMW_SRC_DIGEST = "4adaedf157834c0e"
# DRAM bytes of one zopt_ns_orthogonalize_many call over the 48-matrix stress set (dram__bytes_read.sum
# + dram__bytes_write.sum summed over its launches, one ncu pass on the full set), valid while
# the Newton-Schulz sources hash to NS_SRC_DIGEST
NS_SOURCES = ("ns.cu", "ns_gemm.cu", "ns_prep.cu", "ns_tile.cuh", "tc.cuh", "launch.cuh", "norm_impl.cuh")
NS_TRAFFIC_PER_CALL = 258872122112 + 39090095616
NS_SRC_DIGEST = "4cb7bb9b25d943a4"
MICRO_STEPS = 4
ACC_BYTES = 6 + 10 * (MICRO_STEPS - 1)  # first part: read bf16 2 + write fp32 4; later: + read fp32 4
# two parts to a pass: the first pair reads 2 x 2 and writes 4; each later pair also reads the sum
PAIRED_ACC_BYTES = 8 + 12 * (MICRO_STEPS // 2 - 1)
BF16_STEP_BYTES = 2 + 28  # norm reads the bf16 gradient; the step reads p, m, v, g (14) and writes p, m, v, bf16 (14)


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


def source_digest(files) -> str:
    """The first 16 hex digits of the sha256 of the named kernel sources, in order."""
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "zero_sharded_optimizer_flat_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def adamw_traffic(S: int):
    """DRAM bytes per adamw_kernel launch over S elements from the committed ncu capture, or
    None if the kernel's sources changed since."""
    ok = source_digest(("adamw.cu", "adam_common.cuh", "internal.h", "launch.cuh")) == ADAMW_SRC_DIGEST
    return round(ADAMW_TRAFFIC_PER_ELEM * S) if ok else None


def ns_traffic(ns) -> int | None:
    """DRAM bytes of one Newton-Schulz call over the whole 48-matrix stress set from the committed
    ncu capture (all 18 launches), or None for another set or if the kernels' sources changed."""
    if ns is None or ns.which != "c5" or sum(G.shape[0] for G, _ in ns.groups) != 48:
        return None
    return NS_TRAFFIC_PER_CALL if source_digest(NS_SOURCES) == NS_SRC_DIGEST else None


def ns_flops(rows: int, cols: int, steps: int) -> float:
    """Algorithmic flops of one call, symmetric halves counted once: per step
    m(m+1)n (X X') + m^2(m+1) (A A') + 2 m^2 n (B X), with m <= n."""
    m, n = min(rows, cols), max(rows, cols)
    return float(steps) * (m * (m + 1) * n + m * m * (m + 1) + 2 * m * m * n)


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the CPU baselines."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


# The AdamW-part oracle over whole shards on every host core. The shard is cut into one
# contiguous slice per core, each stepped by its own spawned process with the oracle's functions
# unchanged (the step is element-wise). The clip coefficient needs the whole shard's sum of
# squares, so every step the processes add their slices' sums through shared memory in a fixed
# order (what W ranks' all-reduce would do) before any of them steps.

def _adamw_oracle_worker(wid, nw, jobs, barrier, sums, marks):
    os.environ["OMP_NUM_THREADS"] = os.environ["OPENBLAS_NUM_THREADS"] = "1"
    import numpy as np
    import torch

    torch.set_num_threads(1)
    import workloads
    from oracle import adamw as OA
    from oracle import clip as OC
    from oracle.accum import accumulate
    from oracle.bf16 import f32_to_bf16_bits

    for j, job in enumerate(jobs):
        S = job["S"]
        lo, hi = S * wid // nw, S * (wid + 1) // nw
        n = hi - lo
        seed = job["seed"]
        p = workloads.shard_vector(n, 0.02, seed, 1 + 1000 * wid).numpy()
        m = np.zeros(n, np.float32)
        v = np.zeros(n, np.float32)
        mask = np.ones(n, np.uint8)
        mask[(-lo) % 1000::1000] = 0  # a synthetic decay mask: every 1000th shard slot excluded
        micro = [workloads.shard_vector(n, 1e-3, seed, 2 + k + 1000 * wid, dtype=torch.bfloat16).float().numpy()
                 for k in range(job["micro"])]
        h = OA.Hyper(job["lr"], job["beta1"], job["beta2"], job["eps"], job["weight_decay"])
        t = 0
        for it in range(job["warmup"] + job["steps"]):
            if it == job["warmup"]:
                barrier.wait()
                marks[2 * (j * nw + wid)] = time.perf_counter()
            g = accumulate(micro) if len(micro) > 1 else micro[0]
            sums[wid] = OC.sumsq(g)
            barrier.wait()
            total = sum(sums[k] for k in range(nw))
            barrier.wait()
            st = OC.clip_from_sumsq(total, job["max_norm"])
            t += 1
            OA.step_flat_f32(p, m, v, g, mask, st["clip_coef"], h, t)
            f32_to_bf16_bits(p)
        marks[2 * (j * nw + wid) + 1] = time.perf_counter()
        del p, m, v, micro


def adamw_oracle_on_all_cores(jobs: list) -> list:
    """Runs each job (a shard of S elements, `micro` bf16 micro-step gradients, `warmup` untimed
    and `steps` timed steps) through the AdamW-part oracle on every host core; returns, per job,
    the whole-job seconds of its timed steps (first start to last finish over the processes)."""
    import multiprocessing as mp
    nw = os.cpu_count() or 1
    ctx = mp.get_context("spawn")  # never fork a process that holds a CUDA context
    barrier = ctx.Barrier(nw)
    sums = ctx.Array("d", nw, lock=False)
    marks = ctx.Array("d", 2 * nw * len(jobs), lock=False)
    procs = [ctx.Process(target=_adamw_oracle_worker, args=(k, nw, jobs, barrier, sums, marks)) for k in range(nw)]
    for pr in procs:
        pr.start()
    for pr in procs:
        pr.join()
    if any(pr.exitcode != 0 for pr in procs):
        raise RuntimeError("an AdamW oracle process failed")
    out = []
    for j in range(len(jobs)):
        starts = [marks[2 * (j * nw + k)] for k in range(nw)]
        ends = [marks[2 * (j * nw + k) + 1] for k in range(nw)]
        out.append(max(ends) - min(starts))
    return out


def adamw_job(name: str, steps: int, warmup: int) -> dict:
    """The AdamW part of a parameter set's step as the oracle runs it: the set's whole rank-r
    shard, its micro-steps summed in fp32, norm/clip, AdamW, bf16 round-out."""
    import workloads
    from oracle.layout import shard_len
    w = workloads.get(name)
    S = shard_len([p.numel for p in w.adamw], w.bucket, w.world)
    return {"name": name, "S": S, "micro": max(1, w.micro_steps), "seed": w.seed, "lr": w.lr, "beta1": w.beta1,
            "beta2": w.beta2, "eps": w.eps, "weight_decay": w.weight_decay, "max_norm": w.max_norm,
            "steps": steps, "warmup": warmup,
            "bytes_per_element": ACC_BYTES + ADAMW_BYTES if w.micro_steps > 1 else BF16_STEP_BYTES}


def ns_oracle_rates() -> dict:
    """The fp64 Newton-Schulz oracle (numpy, the host's threaded BLAS) on whole matrix sets: the
    tiny decoder's 8 matrices, the GPT-2-small body's 48, the 1.1B set's 12 rank-0 matrices, the
    stress set's 256 x 1024 block and one whole 4096 x 4096 stress matrix. The whole stress set's
    time is extrapolated from the measured rate of that 4096^2 matrix (labelled so)."""
    import numpy as np
    import torch

    import workloads
    from oracle.ns import newton_schulz

    def timed(mats, reps=1):
        t0 = time.perf_counter()
        for _ in range(reps):
            for x in mats:
                newton_schulz(x, steps=5)
        return (time.perf_counter() - t0) / reps

    def sets(name):
        w = workloads.get(name)
        ps = w.owned_muon() if w.world > 1 else w.muon
        return [workloads.ns_input(p.shape[0], p.shape[1], w.seed, 600 + i, dtype=torch.bfloat16)
                .float().numpy().astype(np.float64) for i, p in enumerate(ps)]

    out = {}
    for name, label in (("c1", "tiny decoder, 8 matrices"), ("c2", "GPT-2-small body, 48 matrices"),
                        ("c3", "1.1B set, rank 0 of 8, 12 matrices")):
        mats = sets(name)
        fl = sum(ns_flops(x.shape[0], x.shape[1], 5) for x in mats)
        sec = timed(mats, 3 if name == "c1" else 1)
        out[name] = {"what": label, "s": round(sec, 4), "tflops": round(fl / sec / 1e12, 4)}
    blk = [workloads.ns_input(256, 1024, 5, 0, dtype=torch.bfloat16).float().numpy().astype(np.float64)]
    sec = timed(blk, 5)
    out["c5_block"] = {"what": "stress set's 256x1024 block", "s": round(sec, 4),
                       "tflops": round(ns_flops(256, 1024, 5) / sec / 1e12, 4)}
    big = [workloads.ns_input(4096, 4096, 5, 1, dtype=torch.bfloat16, frobenius_normalise=True)
           .float().numpy().astype(np.float64)]
    sec = timed(big)
    rate = ns_flops(4096, 4096, 5) / sec
    stress = 16 * (ns_flops(4096, 4096, 5) + 2 * ns_flops(4096, 14336, 5))
    out["c5_4096"] = {"what": "one whole 4096x4096 stress matrix", "s": round(sec, 4),
                      "tflops": round(rate / 1e12, 4)}
    out["c5_whole_extrapolated"] = {"what": "the whole 48-matrix stress set, EXTRAPOLATED from the 4096^2 "
                                            "matrix's rate", "s": round(stress / rate, 1)}
    return out


def cpu_baselines() -> tuple:
    """The GPU arm's CPU baselines: the AdamW-part oracle on every core over the whole shard of
    each parameter set (two timed steps after one untimed), and the fp64 Newton-Schulz oracle."""
    names = ["c4", "c1", "c2", "c3"]
    jobs = [adamw_job(nm, 2, 1) for nm in names]
    S = jobs[0]["S"]
    secs = adamw_oracle_on_all_cores(jobs)
    cores, model = os.cpu_count(), cpu_model()
    per = {}
    for job, sec in zip(jobs, secs):
        per[job["name"]] = {"shard_len": job["S"], "bytes_per_element": job["bytes_per_element"],
                            "ms_per_step": round(sec / job["steps"] * 1e3, 2),
                            "value": round(job["bytes_per_element"] * job["S"] * job["steps"] / sec / 1e9, 3),
                            "unit": "GB/s"}
    main = per["c4"]
    cpu = {"value": main["value"], "unit": "GB/s", "cores": cores, "cpu_model": model, "kind": "oracle",
           "sample": f"the whole {S:,}-element shard (2e9-parameter set, rank 0 of 8): 4 bf16 micro-steps summed "
                     "in fp32 + norm/clip + AdamW + bf16 round-out, numpy fp32 exact-order oracle, 2 timed steps "
                     f"after 1 untimed, one process per core ({cores}) each stepping a 1/{cores} slice, the slices' "
                     "sums of squares added every step",
           "per_config": per}
    ns_t0 = time.perf_counter()
    ns = ns_oracle_rates()
    cpu_ns = {"value": ns["c5_4096"]["tflops"], "unit": "TFLOP/s", "cores": cores, "cpu_model": model,
              "kind": "oracle",
              "sample": "fp64 Newton-Schulz (5 steps) on one whole 4096x4096 stress matrix, numpy with the host's "
                        f"threaded BLAS ({time.perf_counter() - ns_t0:.1f} s for all the sets below)",
              "per_config": ns}
    return cpu, cpu_ns


def run_reference(args, rank: int) -> None:
    """The oracle as it stands, on the host's cores: `--warmup` untimed then `--steps` timed steps.
    A step is the AdamW part over the whole 2e9-parameter shard on every core (the processes add
    their slices' sums of squares each step) and one fp64 Newton-Schulz call on a whole 4096 x 4096
    stress matrix (numpy's threaded BLAS); rank 0 only."""
    if rank != 0:
        return
    import numpy as np
    import torch

    import workloads
    from oracle.ns import newton_schulz

    job = adamw_job("c4", args.steps, args.warmup)
    if args.ref_elements > 0:  # a shorter prefix of the shard (quick checks of the line)
        job["S"] = min(job["S"], args.ref_elements)
    ta = adamw_oracle_on_all_cores([job])[0]
    nsz = args.ref_ns_size
    x = workloads.ns_input(nsz, nsz, 5, 1, dtype=torch.bfloat16, frobenius_normalise=True)\
        .float().numpy().astype(np.float64)
    for _ in range(args.warmup):
        newton_schulz(x, steps=5)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        newton_schulz(x, steps=5)
    tn = time.perf_counter() - t0
    K = args.steps
    S = job["S"]
    value = round(job["bytes_per_element"] * S * K / ta / 1e9, 3)
    cores, model = os.cpu_count(), cpu_model()
    cpu = {"value": value, "unit": "GB/s", "cores": cores, "cpu_model": model, "kind": "oracle",
           "sample": f"{K} timed steps after {args.warmup} warm-up steps; each step: the AdamW-part oracle "
                     f"(4-micro-step fp32 accumulation + norm/clip + AdamW + bf16 round-out) over the whole {S:,}-"
                     f"element shard ({ta / K * 1e3:.1f} ms, numpy, one process per core each stepping a 1/{cores} "
                     f"slice) and one fp64 Newton-Schulz call (5 steps) on a whole {nsz}x{nsz} stress matrix "
                     f"({tn / K * 1e3:.1f} ms, numpy's threaded BLAS)"}
    fl = ns_flops(nsz, nsz, 5)
    ns = {"value": round(fl * K / tn / 1e12, 5), "unit": "TFLOP/s", "cores": cores, "cpu_model": model,
          "kind": "oracle",
          "sample": f"{K} timed fp64 Newton-Schulz calls (5 steps) on a whole {nsz}x{nsz} stress matrix ({tn:.2f} s)"}
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": K, "warmup": args.warmup, "ms_per_step": round((ta + tn) / K * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "l2": "inputs larger than L2"},
            "adamw_part": {"ms": round(ta / K * 1e3, 3), "bytes_per_element": job["bytes_per_element"],
                           "elements": S},
            "ns": {"value": ns["value"], "unit": "TFLOP/s", "ms_per_step": round(tn / K * 1e3, 3)},
            "cpu_baseline": cpu, "cpu_baseline_ns": ns,
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


class NsPart:
    """A Newton-Schulz set (the stress set or the GPT-2-small body): bf16 matrices, one call over all shapes."""

    def __init__(self, Z, torch, seed: int, steps: int, count_limit: int = 0, which: str = "c5"):
        import workloads
        self.Z, self.steps, self.which = Z, steps, which
        w = workloads.get(which)
        shapes = []
        for prm in w.muon:
            if prm.shape not in shapes:
                shapes.append(prm.shape)
        self.groups = []
        gen = torch.Generator(device="cuda").manual_seed(seed)
        for (r, c) in shapes:
            count = sum(1 for prm in w.muon if prm.shape == (r, c))
            if count_limit > 0:
                count = min(count, count_limit)
            G = torch.randn(count, r, c, device="cuda", generator=gen)
            if which == "c5":
                G /= torch.linalg.vector_norm(G, dim=(1, 2), keepdim=True)  # Frobenius-normalised
            else:
                G *= 1e-3  # gradient-like scale
            G = G.to(torch.bfloat16)
            self.groups.append((G, torch.empty_like(G)))
        # one call over every shape (zopt_ns_orthogonalize_many): each shape's whole batch is one
        # group; shapes below 1024 share persistent fused launches (six to a launch)
        self.ws = Z.new_ns_workspace_many([(G.shape[1], G.shape[2], G.shape[0]) for G, _ in self.groups])
        # the end-to-end pass calls zopt_ns_orthogonalize on chunks of each shape: at least 4
        # matrices and up to ~48 MB of input (small matrices: fewer calls, each bound by its
        # chain of dependent products rather than by its size), or two such chunks merged
        self.per_chunk = []
        for G, _ in self.groups:
            cap = min(G.shape[0], max(4, (48 << 20) // (G[0].numel() * G.element_size())))
            pieces = -(-G.shape[0] // cap)
            self.per_chunk.append(-(-G.shape[0] // pieces))  # even pieces
        self.ws_chunk = torch.empty(max(Z.ns_workspace(G.shape[1], G.shape[2], min(G.shape[0], 2 * per))
                                        for (G, _), per in zip(self.groups, self.per_chunk)),
                                    dtype=torch.uint8, device="cuda")
        self.flops = sum(ns_flops(G.shape[1], G.shape[2], steps) * G.shape[0] for G, _ in self.groups)
        fused = sum(1 for G, _ in self.groups if min(G.shape[1], G.shape[2]) < 1024)
        # the norm of every matrix in one launch (bf16 input), then one scaling launch if any
        # shape is wide or square and one transpose launch if any is tall (at most 16 shapes
        # to a launch); then one fused launch per six small shapes, and for the large ones each
        # product of a step in one launch per four shapes
        wide = sum(1 for G, _ in self.groups if G.shape[1] <= G.shape[2])
        tall = len(self.groups) - wide
        prep = -(-len(self.groups) // 16) + -(-wide // 16) + -(-tall // 16)
        large = len(self.groups) - fused
        self.launches = prep + -(-fused // 6) + 3 * steps * -(-large // 4)
        names = (["ns_fused_kernel (X X', B', B'X of every step, shapes below 1024)"] if fused else []) + \
                (["gemm_bf16_pair_kernel (X X', B', B'X on CTA pairs)"] if fused < len(self.groups) else [])
        self.kernel = " + ".join(names)

    def run(self, stream):
        self.Z.ns_orthogonalize_many(self.groups, self.ws, steps=self.steps, stream=stream)


class MuonPart:
    """One Muon step over a parameter set's Muon matrices that rank 0 owns (round-robin by index,
    the set's W): for the 1.1B Llama-style set (W = 8) 4 x 2048^2, 4 x 2048x512, 4 x 2048x11264;
    for the GPT-2-small body (W = 1) all 48. bf16 gradients ~N(0, 1e-3), masters ~N(0, 0.02)."""

    def __init__(self, Z, torch, seed: int, which: str = "c3"):
        import workloads
        self.Z = Z
        w = workloads.get(which)
        shapes = {}
        for prm in w.owned_muon():
            shapes[prm.shape] = shapes.get(prm.shape, 0) + 1
        gen = torch.Generator(device="cuda").manual_seed(seed)
        self.jobs = []
        for (r, c), b in shapes.items():
            p = torch.randn(b, r, c, device="cuda", generator=gen).mul_(0.02)
            g = torch.randn(b, r, c, device="cuda", generator=gen).mul_(1e-3).to(torch.bfloat16)
            self.jobs.append((p, torch.zeros_like(p), g, torch.empty(b, r, c, dtype=torch.int16, device="cuda"),
                              Z.new_muon_stats(b)))
        self.ws = Z.new_muon_workspace_many([(r, c, b) for (r, c), b in shapes.items()])
        self.count = sum(shapes.values())
        self.flops = sum(ns_flops(r, c, 5) * b for (r, c), b in shapes.items())
        n = sum(r * c * b for (r, c), b in shapes.items())
        # per element: momentum 12 (bf16 grad in; buf in and out; u out in bf16) and update 12
        # (master in and out, bf16 U in, bf16 weights out); U's statistics come from the last
        # Newton-Schulz product's epilogue, u's norm from the momentum pass
        self.bytes = 24 * n
        owner = f"owned by rank 0 of {w.world}" if w.world > 1 else "(W = 1)"
        self.what = (f"{self.count} matrices {sorted(shapes)} of the {which} set {owner}, "
                     "zopt_muon_step_many, 5 Newton-Schulz steps")
        self.lr = w.muon_lr

    def run(self, stream):
        self.Z.muon_step_many(self.jobs, self.ws, lr=self.lr, stream=stream)


def config_lines(Z, torch, stream, pk, K: int) -> dict:
    """The smaller parameter sets, each timed apart (3 untimed then K timed iterations, CUDA
    events on the launching stream): the tiny decoder (1,048,832-element shard), the GPT-2-small
    set (38,652,672) and the 1.1B set's rank 0 of 8 (8,200,448) take norm/clip and the AdamW step
    on a bf16 gradient (30 B/element; the adamw_kernel alone 28 B), as two calls and as the one
    call zopt_adamw_clip_step, with a 256 MB L2 flush between
    iterations, except the tiny set, which is timed L2-resident and makes no roofline claim; the
    tiny decoder's and the GPT-2-small body's Newton-Schulz sets, and the GPT-2-small body's Muon
    step, against the burst bf16 peak (each call lasts about a millisecond; at least 300 calls
    are timed, with the SM clock sampled)."""
    import statistics as stats_

    import workloads
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    res = {}
    for name in ("c1", "c2", "c3"):
        w = workloads.get(name)
        lay = Z.ShardLayout([p.numel for p in w.adamw], [p.decay for p in w.adamw], w.bucket, w.world, w.rank)
        S = lay.shard_len
        table = lay.device_table()
        gen = torch.Generator(device="cuda").manual_seed(w.seed)
        p = torch.randn(S, device="cuda", generator=gen).mul_(0.02)
        m, v = torch.zeros(S, device="cuda"), torch.zeros(S, device="cuda")
        g = torch.randn(S, device="cuda", generator=gen).mul_(1e-3).to(torch.bfloat16)
        out = torch.empty(S, dtype=torch.int16, device="cuda")
        clip, state, ws = Z.new_clip_stats(), Z.new_adam_state(), Z.new_norm_workspace(S)
        resident = name == "c1"
        evs = [(mk(), mk(), mk()) for _ in range(3 + K)]
        for i, (e0, e1, e2) in enumerate(evs):
            if not resident:
                flush.zero_()
            e0.record(stream)
            Z.grad_norm_clip(g, w.max_norm, ws, clip, stream=stream)
            e1.record(stream)
            Z.adamw_step(lay, table, p, m, v, g, out, lr=w.lr_at(i % w.steps), beta1=w.beta1, beta2=w.beta2,
                         eps=w.eps, weight_decay=w.weight_decay, clip_stats=clip, adam_state=state, stream=stream)
            e2.record(stream)
        torch.cuda.synchronize()
        step_ms = stats_.mean(e0.elapsed_time(e2) for e0, _, e2 in evs[3:])
        kern_ms = stats_.mean(e1.elapsed_time(e2) for _, e1, e2 in evs[3:])
        part = BF16_STEP_BYTES * S / (step_ms * 1e-3) / 1e9
        kern = 28 * S / (kern_ms * 1e-3) / 1e9
        entry = {"shard_len": S, "world": w.world,
                 "adamw_part": {"what": "zopt_grad_norm_clip + zopt_adamw_step, bf16 gradient", "ms": round(step_ms, 4),
                                "bytes_per_element": BF16_STEP_BYTES, "achieved": round(part, 1), "unit": "GB/s"},
                 "l2": "L2-resident (the whole state fits in L2): no roofline claim" if resident
                       else "256 MB L2 flush between iterations"}
        if not resident:
            entry["adamw_part"]["frac"] = round(part / pk["hbm_gbs"], 4)
            entry["roofline"] = {"kernel": "adamw_kernel (bf16 gradient)", "bound": "hbm", "achieved": round(kern, 1),
                                 "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(kern / pk["hbm_gbs"], 4),
                                 "bytes_per_element": 28, "avg_launch_ms": round(kern_ms, 4)}
        else:
            entry["adamw_kernel"] = {"ms": round(kern_ms, 4), "achieved": round(kern, 1), "unit": "GB/s"}
        # the same step through zopt_adamw_clip_step: the norm / clip reduction and the update in
        # one launch (same bytes; the gradient's second read from L2 only where it survives the update's stream)
        cws = Z.new_adamw_clip_workspace(S)
        evs = [(mk(), mk()) for _ in range(3 + K)]
        for i, (e0, e1) in enumerate(evs):
            if not resident:
                flush.zero_()
            e0.record(stream)
            Z.adamw_clip_step(lay, table, p, m, v, g, out, lr=w.lr_at(i % w.steps), max_norm=w.max_norm, ws=cws,
                              clip_stats=clip, adam_state=state, beta1=w.beta1, beta2=w.beta2, eps=w.eps,
                              weight_decay=w.weight_decay, stream=stream)
            e1.record(stream)
        torch.cuda.synchronize()
        fused_ms = stats_.mean(e0.elapsed_time(e1) for e0, e1 in evs[3:])
        fused = BF16_STEP_BYTES * S / (fused_ms * 1e-3) / 1e9
        entry["adamw_clip_step"] = {"what": "zopt_adamw_clip_step (the same step in one launch)",
                                    "ms": round(fused_ms, 4), "bytes_per_element": BF16_STEP_BYTES,
                                    "achieved": round(fused, 1), "unit": "GB/s"}
        if not resident:
            entry["adamw_clip_step"]["frac"] = round(fused / pk["hbm_gbs"], 4)
        res[name] = entry
        del p, m, v, g, out, ws, cws

    def timed_calls(run):
        # calls of about a millisecond: at least 300 of them (~0.3 s) so that the clock sampler
        # sees a few readings
        for _ in range(3):
            run(stream)
        torch.cuda.synchronize()
        evs = [(mk(), mk()) for _ in range(max(K, 300))]
        with Clocks(smi_id(torch.cuda.current_device())) as clk_c:
            for a, b in evs:
                a.record(stream)
                run(stream)
                b.record(stream)
            torch.cuda.synchronize()
        return stats_.mean(a.elapsed_time(b) for a, b in evs), clk_c.summary()

    for name in ("c1", "c2"):
        nsp = NsPart(Z, torch, 9000, 5, 0, name)
        ms_, clk_ = timed_calls(nsp.run)
        tf = nsp.flops / (ms_ * 1e-3) / 1e12
        res[name]["ns"] = {"what": f"{sum(G.shape[0] for G, _ in nsp.groups)} bf16 matrices "
                                   f"{[tuple(G.shape[1:]) for G, _ in nsp.groups]}, one zopt_ns_orthogonalize_many "
                                   "call, 5 steps", "ms": round(ms_, 4), "achieved": round(tf, 1), "unit": "TFLOP/s",
                           "peak": pk["bf16_tflops"], "frac": round(tf / pk["bf16_tflops"], 4),
                           "peak_source": pk["source"] + " bf16 burst", "calls_timed": max(K, 300), "clocks": clk_}
        if name == "c1":
            res[name]["ns"]["note"] = "the set is 3.4 MB (L2-resident) and latency-bound: no roofline claim"
        del nsp
    mu2 = MuonPart(Z, torch, 9100, "c2")
    ms_, clk_ = timed_calls(mu2.run)
    tf = mu2.flops / (ms_ * 1e-3) / 1e12
    res["c2"]["muon_step"] = {"what": mu2.what, "ms": round(ms_, 4), "ns_equivalent_tflops": round(tf, 1),
                              "peak": pk["bf16_tflops"], "frac": round(tf / pk["bf16_tflops"], 4),
                              "peak_source": pk["source"] + " bf16 burst",
                              "calls_timed": max(K, 300), "clocks": clk_,
                              "note": "the whole step's time against the Newton-Schulz flops alone"}
    del mu2
    torch.cuda.empty_cache()
    return res


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
    parts = set(args.parts.split(","))
    stream = torch.cuda.current_stream()
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    mean = lambda evs: statistics.mean(a.elapsed_time(b) for a, b in evs)  # noqa: E731

    # ---- part 1: micro-step accumulation with fused clip stats + AdamW over this rank's shard
    w = workloads.get("c4")
    sim_rank = rank % w.world
    lay = Z.ShardLayout([p.numel for p in w.adamw], [p.decay for p in w.adamw], w.bucket, w.world, sim_rank)
    S = lay.shard_len if args.shard_len <= 0 else min(args.shard_len, lay.shard_len)
    if S != lay.shard_len:  # a prefix of the same parameter list, as its own layout
        lay = Z.ShardLayout([S], [1], 1 << 40, 1, 0)
    if "adamw" in parts:
        table = lay.device_table()
        gen = torch.Generator(device="cuda").manual_seed(w.seed * 100 + sim_rank)
        p = torch.randn(S, device="cuda", generator=gen).mul_(0.02)
        m = torch.zeros(S, device="cuda")
        v = torch.zeros(S, device="cuda")
        micro = [torch.randn(S, device="cuda", generator=gen).mul_(1e-3).to(torch.bfloat16)
                 for _ in range(MICRO_STEPS)]
        g = torch.empty(S, device="cuda")  # the fp32 shard gradient (sum of the micro-steps)
        out = torch.empty(S, dtype=torch.int16, device="cuda")
        clip, state = Z.new_clip_stats(), Z.new_adam_state()
        ws = Z.new_norm_workspace(S)
        kw = dict(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, weight_decay=w.weight_decay, clip_stats=clip,
                  adam_state=state)
    # ---- part 2: Newton-Schulz over the stress set (whole matrices owned by this rank)
    ns = NsPart(Z, torch, 5000 + rank, 5, args.ns_count, "c5" if args.ns_set == "stress" else "c2") \
        if "ns" in parts else None

    K = args.steps
    ev_a = [(mk(), mk()) for _ in range(K)]   # accumulation + clip + AdamW part
    ev_k = [(mk(), mk()) for _ in range(K)]   # adamw_kernel alone
    ev_n = [(mk(), mk()) for _ in range(K)]   # Newton-Schulz part

    def adamw_part(i=None):
        for k, mg in enumerate(micro):
            Z.grad_accumulate(g, mg, first=k == 0, last=k == MICRO_STEPS - 1, max_norm=w.max_norm, ws=ws,
                              stats=clip, stream=stream)
        if i is not None:
            ev_k[i][0].record(stream)
        Z.adamw_step(lay, table, p, m, v, g, out, stream=stream, **kw)
        if i is not None:
            ev_k[i][1].record(stream)

    def step(i=None):
        if "adamw" in parts:
            if i is not None:
                ev_a[i][0].record(stream)
            adamw_part(i)
            if i is not None:
                ev_a[i][1].record(stream)
        if ns is not None:
            if i is not None:
                ev_n[i][0].record(stream)
            ns.run(stream)
            if i is not None:
                ev_n[i][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0, t1 = mk(), mk()
    with Clocks(smi_id(local_rank)) as clk:
        # every launch of the timed steps is queued behind a device-side delay, so the events
        # time GPU execution only, not the host's enqueue rate (dmuon PR #16's timing method)
        torch.cuda._sleep(int(args.prequeue_ms * 2.0e6))
        t0.record(stream)
        for i in range(K):
            step(i)
        t1.record(stream)
        torch.cuda.synchronize()
    clocks = clk.summary()
    ms = t0.elapsed_time(t1) / K
    a_ms = mean(ev_a) if "adamw" in parts else 0.0
    k_ms = mean(ev_k) if "adamw" in parts else 0.0
    n_ms = mean(ev_n) if ns is not None else 0.0
    # the stand-alone norm / clip / found_inf reduction (zopt_grad_norm_clip, for a gradient that
    # arrives already summed) over the same fp32 shard gradient (4 B/element, > L2), timed apart
    # from the steps
    nr_ms = 0.0
    if "adamw" in parts:
        nstats = Z.new_clip_stats()
        for _ in range(3):
            Z.grad_norm_clip(g, w.max_norm, ws, nstats, stream=stream)
        torch.cuda.synchronize()
        ev_r = [(mk(), mk()) for _ in range(max(K, 3))]
        for a_ev, b_ev in ev_r:
            a_ev.record(stream)
            Z.grad_norm_clip(g, w.max_norm, ws, nstats, stream=stream)
            b_ev.record(stream)
        torch.cuda.synchronize()
        nr_ms = mean(ev_r)
    # the same step with the micro-steps summed two to a pass (zopt_grad_accumulate2: bit for bit
    # the four single passes, 20 instead of 36 B/element for the sum), timed apart
    pa_ms = 0.0
    if "adamw" in parts:
        def paired_part():
            for k in range(0, MICRO_STEPS, 2):
                Z.grad_accumulate2(g, micro[k], micro[k + 1], first=k == 0, last=k + 2 == MICRO_STEPS,
                                   max_norm=w.max_norm, ws=ws, stats=clip, stream=stream)
            Z.adamw_step(lay, table, p, m, v, g, out, stream=stream, **kw)
        for _ in range(3):
            paired_part()
        torch.cuda.synchronize()
        ev_p = [(mk(), mk()) for _ in range(max(K, 3))]
        for a_ev, b_ev in ev_p:
            a_ev.record(stream)
            paired_part()
            b_ev.record(stream)
        torch.cuda.synchronize()
        pa_ms = mean(ev_p)
    # zopt_adamw_rescale_step (re-target the step just taken to another gradient scale) over the
    # shard: 30 B/element like the step itself, timed apart
    rs_ms = 0.0
    if "adamw" in parts:
        rkw = dict(kw, clip_stats=None)
        for _ in range(3):
            Z.adamw_rescale_step(lay, p, m, v, g, out, old_scale=1.0, new_scale=0.5, stream=stream, **rkw)
        torch.cuda.synchronize()
        ev_s = [(mk(), mk()) for _ in range(max(K, 3))]
        for a_ev, b_ev in ev_s:
            a_ev.record(stream)
            Z.adamw_rescale_step(lay, p, m, v, g, out, old_scale=1.0, new_scale=0.5, stream=stream, **rkw)
            b_ev.record(stream)
        torch.cuda.synchronize()
        rs_ms = mean(ev_s)
    # one Muon step (zopt_muon_step_many: momentum, Newton-Schulz, statistics, guarded update,
    # bf16 round-out) over the matrices rank 0 of the 1.1B Llama-style set owns, timed apart
    mu_ms, mu = 0.0, None
    mu_clocks = None
    if "muon" in parts:
        # ~3 ms a step: 200 steps (~0.6 s, 2.7 GB touched a step, far above L2) give the clock
        # sampler a few readings
        mu = MuonPart(Z, torch, 7000 + rank)
        for _ in range(3):
            mu.run(stream)
        torch.cuda.synchronize()
        ev_m = [(mk(), mk()) for _ in range(max(K, 200))]
        with Clocks(smi_id(local_rank)) as clk_m:
            for a_ev, b_ev in ev_m:
                a_ev.record(stream)
                mu.run(stream)
                b_ev.record(stream)
            torch.cuda.synchronize()
        mu_clocks = clk_m.summary()
        mu_ms = mean(ev_m)
    # the smaller parameter sets (tiny decoder, GPT-2-small, the 1.1B set's rank 0), timed apart
    cfg = config_lines(Z, torch, stream, peaks(), max(K, 3)) if "configs" in parts and rank == 0 else None
    if dist:
        tt = torch.tensor([ms, a_ms, k_ms, n_ms, nr_ms, rs_ms, mu_ms], device="cuda")
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        ms, a_ms, k_ms, n_ms, nr_ms, rs_ms, mu_ms = (float(x) for x in tt)
        dist.barrier()

    # ---- end to end through the public API with host buffers: each part takes its inputs
    # (the micro-step gradients; the Newton-Schulz inputs) from pinned host memory and reads
    # its results back to pinned host memory (the clip stats and the bf16 compute weights; the
    # orthogonalised matrices). The accumulation passes read the pinned micro-step gradients
    # themselves, over the CPU-GPU link (no staging copy); the bf16 weights go back on a copy
    # stream while the next step's accumulation reads its gradients (the link is full duplex),
    # and a step's AdamW launch waits for the previous read-back of the weights it overwrites.
    # The Newton-Schulz inputs and outputs move on two copy streams, overlapped with the compute
    # of the previous or next matrix group. Each part runs its steps back to back and is timed
    # from its first transfer to its last read-back, divided by the steps (steady state).
    h2d = d2h = 0
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    if "adamw" in parts:
        micro_host = [mg.cpu().pin_memory() for mg in micro]
        stats_host = torch.empty(Z.CLIP_STATS_BYTES, dtype=torch.uint8).pin_memory()
        out_host = torch.empty(S, dtype=torch.int16).pin_memory()
        out_read = ev()
        out_read.record(stream)
        h2d += 2 * S * MICRO_STEPS
        d2h += Z.CLIP_STATS_BYTES + 2 * S
    if ns is not None:
        ns_host = [(G.cpu().pin_memory(), torch.empty(X.shape, dtype=X.dtype).pin_memory()) for G, X in ns.groups]
        h2d += sum(G.numel() * 2 for G, _ in ns.groups)
        d2h += sum(X.numel() * 2 for _, X in ns.groups)
        # chunks of ns.per_chunk matrices: the two smallest go first and last (only their upload
        # and read-back are not overlapped); in between, neighbouring chunks of one shape are
        # merged into calls of up to twice as many matrices (their transfers hide behind compute,
        # and a larger call fills the GPU better), largest first
        spans = [(gi, lo, min(G.shape[0], lo + ns.per_chunk[gi])) for gi, (G, _) in enumerate(ns.groups)
                 for lo in range(0, G.shape[0], ns.per_chunk[gi])]
        size = lambda sp: (sp[2] - sp[1]) * ns.groups[sp[0]][0][0].numel()  # noqa: E731
        spans.sort(key=size)
        if len(spans) > 1:
            mid = []
            for sp in sorted(spans[2:]):
                gi = sp[0]
                if mid and mid[-1][0] == gi and mid[-1][2] == sp[1] and sp[2] - mid[-1][1] <= 2 * ns.per_chunk[gi]:
                    mid[-1] = (gi, mid[-1][1], sp[2])
                else:
                    mid.append(sp)
            spans = [spans[0]] + sorted(mid, key=size, reverse=True) + [spans[1]]
        chunks = [(ns.groups[gi][0][lo:hi], ns.groups[gi][1][lo:hi], ns_host[gi][0][lo:hi], ns_host[gi][1][lo:hi])
                  for gi, lo, hi in spans]
        ns_done = [ev() for _ in chunks]
        out_done = [ev() for _ in chunks]
        for e in ns_done + out_done:
            e.record(stream)
    e2e_steps = max(3, min(K, 6))

    def e2e_adamw_step():
        for k, mh in enumerate(micro_host):
            Z.grad_accumulate(g, mh, first=k == 0, last=k == MICRO_STEPS - 1, max_norm=w.max_norm, ws=ws,
                              stats=clip, stream=stream)
        stream.wait_event(out_read)  # the previous step's weights have reached the host
        Z.adamw_step(lay, table, p, m, v, g, out, stream=stream, **kw)
        stats_host.copy_(clip, non_blocking=True)
        done = ev()
        done.record(stream)
        d2h_s.wait_event(done)
        with torch.cuda.stream(d2h_s):
            out_host.copy_(out, non_blocking=True)
        out_read.record(d2h_s)

    def e2e_ns_step():
        start = ev()
        start.record(stream)
        h2d_s.wait_event(start)
        landed = []
        for ci, (G, X, hG, hX) in enumerate(chunks):
            h2d_s.wait_event(ns_done[ci])  # the previous step has read G
            with torch.cuda.stream(h2d_s):
                G.copy_(hG, non_blocking=True)
            e = ev()
            e.record(h2d_s)
            landed.append(e)
        for ci, (G, X, hG, hX) in enumerate(chunks):
            stream.wait_event(landed[ci])
            stream.wait_event(out_done[ci])  # the previous step's X has been read back
            Z.ns_orthogonalize(G, X, ns.ws_chunk, steps=ns.steps, stream=stream)
            ns_done[ci].record(stream)
            d2h_s.wait_event(ns_done[ci])
            with torch.cuda.stream(d2h_s):
                hX.copy_(X, non_blocking=True)
            out_done[ci].record(d2h_s)

    def e2e_leg(one_step, drain):
        for _ in range(2):
            one_step()
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        a_ev, b_ev = mk(), mk()
        a_ev.record(stream)
        for _ in range(e2e_steps):
            one_step()
        for e in drain():
            stream.wait_event(e)
        b_ev.record(stream)
        torch.cuda.synchronize()
        return a_ev.elapsed_time(b_ev) / e2e_steps

    ea_ms = e2e_leg(e2e_adamw_step, lambda: [out_read]) if "adamw" in parts else 0.0
    e2e_clocks = None
    en_ms = 0.0
    if ns is not None:
        with Clocks(smi_id(local_rank)) as clk2:
            en_ms = e2e_leg(e2e_ns_step, lambda: out_done)
        e2e_clocks = clk2.summary()
    if dist:
        tt = torch.tensor([ea_ms, en_ms], device="cuda")
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        ea_ms, en_ms = float(tt[0]), float(tt[1])

    # ---- host cost of one Newton-Schulz call (argument checks, tensor-map encoding, launches),
    # eager and as a replay of the same call captured in a CUDA graph. The calls' GPU work queues
    # behind and is drained afterwards; only the host time is taken here.
    host_ns = None
    if ns is not None:
        reps = 8
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(reps):
            ns.run(stream)
        eager_us = (time.perf_counter() - t0) / reps * 1e6
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            ns.run(torch.cuda.current_stream())
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(reps):
            graph.replay()
        replay_us = (time.perf_counter() - t0) / reps * 1e6
        torch.cuda.synchronize()
        del graph
        host_ns = {"eager_us_per_call": round(eager_us, 1), "graph_replay_us_per_call": round(replay_us, 1),
                   "launches_per_call": ns.launches,
                   "matrices_per_call": sum(G.shape[0] for G, _ in ns.groups)}

    pk = peaks()
    part_bytes = (ACC_BYTES + ADAMW_BYTES) * S
    line = {"metric": METRIC, "n_gpus": world_procs, "steps": K, "warmup": args.warmup,
            "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "shard_len": S, "micro_steps": MICRO_STEPS, "micro_grad_dtype": "bf16",
                       "simulated_world": w.world,
                       "ns_set": (f"{sum(G.shape[0] for G, _ in ns.groups)} bf16 matrices "
                                  f"{[tuple(G.shape[1:]) for G, _ in ns.groups]}, 5 steps") if ns else None,
                       "l2": "inputs larger than L2 (~13 GB touched per step), no flush"}}
    if "adamw" in parts:
        achieved = ADAMW_BYTES * S / (k_ms * 1e-3) / 1e9
        line["value"] = round(part_bytes * world_procs / (a_ms * 1e-3) / 1e9, 2)
        line["unit"] = "GB/s"
        line["adamw_part"] = {"ms": round(a_ms, 4), "bytes_per_element": ACC_BYTES + ADAMW_BYTES,
                              "accumulate_ms": round(a_ms - k_ms, 4), "adamw_kernel_ms": round(k_ms, 4)}
        paired_bytes = PAIRED_ACC_BYTES + ADAMW_BYTES
        line["adamw_part_paired"] = {
            "what": "the same step with the micro-steps summed two to a pass (zopt_grad_accumulate2), timed apart",
            "ms": round(pa_ms, 4), "bytes_per_element": paired_bytes,
            "achieved": round(paired_bytes * S / (pa_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
            "frac": round(paired_bytes * S / (pa_ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4)}
        norm_gbs = 4 * S / (nr_ms * 1e-3) / 1e9
        line["norm_clip"] = {"kernel": "norm_kernel (zopt_grad_norm_clip on the fp32 shard gradient, timed "
                                       "apart from the steps)", "ms": round(nr_ms, 4), "bytes_per_element": 4,
                             "achieved": round(norm_gbs, 1), "unit": "GB/s",
                             "frac": round(norm_gbs / pk["hbm_gbs"], 4)}
        rs_gbs = ADAMW_BYTES * S / (rs_ms * 1e-3) / 1e9
        line["rescale"] = {"kernel": "rescale_kernel (zopt_adamw_rescale_step over the shard, timed apart)",
                           "ms": round(rs_ms, 4), "bytes_per_element": ADAMW_BYTES, "achieved": round(rs_gbs, 1),
                           "unit": "GB/s", "frac": round(rs_gbs / pk["hbm_gbs"], 4)}
        line["roofline_hbm"] = {"kernel": "adamw_kernel", "bound": "hbm", "achieved": round(achieved, 1),
                                "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 4),
                                "traffic": adamw_traffic(S), "peak_source": pk["source"],
                                "algorithmic_bytes_per_launch": ADAMW_BYTES * S, "avg_launch_ms": round(k_ms, 4)}
    if ns is not None:
        tflops = ns.flops / (n_ms * 1e-3) / 1e12
        line["ns"] = {"value": round(tflops * world_procs, 2), "unit": "TFLOP/s", "ms_per_step": round(n_ms, 3),
                      "algorithmic_flops_per_step": ns.flops, "host": host_ns,
                      "tflops_per_sm_mhz": round(tflops / clocks["sm_mhz"], 4) if clocks.get("sm_mhz") else None}
        line["roofline"] = {"kernel": ns.kernel, "bound": "tensor",
                            "achieved": round(tflops, 1), "peak": pk["bf16_tflops_sustained"], "unit": "TFLOP/s",
                            "frac": round(tflops / pk["bf16_tflops_sustained"], 4), "traffic": ns_traffic(ns),
                            "traffic_note": "DRAM bytes of one call (all its launches), from an ncu capture",
                            "peak_source": pk["source"] + " bf16 sustained (the GEMMs run for ~100 ms per step)",
                            "note": "achieved = algorithmic flops of the Newton-Schulz calls / their event time "
                                    "(includes the small normalise/orient kernels)"}
        if "value" not in line:
            line["value"], line["unit"] = line["ns"]["value"], "TFLOP/s"
    elif "adamw" in parts:
        line["roofline"] = line.pop("roofline_hbm")
    if mu is not None:
        line["muon_step"] = {"what": mu.what, "ms": round(mu_ms, 4), "matrices": mu.count,
                             "ns_algorithmic_flops": mu.flops,
                             "ns_equivalent_tflops": round(mu.flops / (mu_ms * 1e-3) / 1e12, 1),
                             "elementwise_bytes": mu.bytes, "steps_timed": max(K, 200), "clocks": mu_clocks,
                             "note": "the whole step's time against the Newton-Schulz flops alone; the momentum and "
                                     "update passes move elementwise_bytes besides (U's statistics come from the last "
                                     "product's epilogue)"}
    line["clocks"] = clocks
    e2e = {"h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    if "adamw" in parts:
        e2e.update(value=round(part_bytes * world_procs / (ea_ms * 1e-3) / 1e9, 2), unit="GB/s",
                   adamw_part_ms=round(ea_ms, 3))
    if ns is not None:
        etf = ns.flops / (en_ms * 1e-3) / 1e12
        e2e.update(ns_value=round(etf * world_procs, 2), ns_unit="TFLOP/s", ns_part_ms=round(en_ms, 3),
                   ns_clocks=e2e_clocks,
                   ns_tflops_per_sm_mhz=round(etf / e2e_clocks["sm_mhz"], 4) if e2e_clocks.get("sm_mhz") else None)
    line["e2e"] = e2e
    if cfg is not None:
        line["configs"] = cfg
    line["gpu_launches"] = K * ((MICRO_STEPS + 1 if "adamw" in parts else 0) + (ns.launches if ns else 0))
    if rank == 0:
        if world_procs == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"], line["cpu_baseline_ns"] = cpu_baselines()
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prequeue-ms", type=float, default=50.0,
                    help="device-side delay (about this many ms at 2 GHz) queued before the timed steps")
    ap.add_argument("--parts", default="adamw,ns,muon,configs",
                    help="comma list: adamw, ns (the timed step), muon (a Muon step timed apart), configs (the "
                         "smaller parameter sets timed apart)")
    ap.add_argument("--ns-set", default="stress", choices=["stress", "gpt2"],
                    help="Newton-Schulz matrices: the 48-matrix 4096-wide stress set, or the GPT-2-small body's 48")
    ap.add_argument("--ns-count", type=int, default=0,
                    help="matrices per Newton-Schulz shape (profiling captures); 0 = the full set of 16")
    ap.add_argument("--ref-elements", type=int, default=0,
                    help="reference arm: step only this many shard elements (quick checks); 0 = the whole shard")
    ap.add_argument("--ref-ns-size", type=int, default=4096,
                    help="reference arm: side of the square stress matrix its Newton-Schulz calls take")
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
