"""Multi-rank host logic on CPU with two gloo ranks (no GPU).

Each rank builds its own view of the flat bucketed layout through the library
(deg/zero.py, ZeroMaster: rank r owns the r-th piece of every bucket) and computes the local
Σg² of its shard of a seeded global gradient with the oracle. The ranks then do the one real
exchange of the step — an all-reduce of the fp64 Σg² (deg/zero.py grad_sq_norm) — and check:

* the shards of all ranks cover every flat element exactly once (the union of the library's
  segments, gathered over gloo);
* the all-reduced Σg² gives the same clip statistics as the whole gradient does.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, numel: list, bucket: int, q) -> None:
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    try:
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        dist.init_process_group("gloo", rank=rank, world_size=world)
        import zero_sharded_optimizer_flat_gb300 as Z
        from oracle import clip as OC

        lay = Z.ShardLayout(numel, None, bucket, world, rank)
        N = sum(numel)
        owned = np.zeros(N, np.int64)
        offsets = np.concatenate([[0], np.cumsum(numel)])
        shard_flat = np.full(lay.shard_len, -1, np.int64)
        for p, po, so, ln in lay.segments():
            f0 = offsets[p] + po
            owned[f0:f0 + ln] += 1
            shard_flat[so:so + ln] = np.arange(f0, f0 + ln)
        t = torch.from_numpy(owned)
        dist.all_reduce(t)  # every flat element owned exactly once over the ranks
        cover_ok = bool(torch.all(t == 1))

        g = np.random.default_rng(7).normal(0, 1e-3, N).astype(np.float32)  # the same on every rank
        local = np.where(shard_flat >= 0, g[np.maximum(shard_flat, 0)], 0).astype(np.float32)
        ss = torch.tensor([OC.sumsq(local)], dtype=torch.float64)
        dist.all_reduce(ss)
        glob = OC.clip_from_sumsq(float(ss[0]), 1e-3)
        ref = OC.clip_stats(g, 1e-3)
        stats_ok = (glob["found_inf"] == ref["found_inf"] and glob["clipped"] == ref["clipped"] and
                    abs(float(glob["clip_coef"]) - float(ref["clip_coef"])) <= 1e-6 * float(ref["clip_coef"]))
        q.put((rank, cover_ok, stats_ok, lay.shard_len))
        dist.destroy_process_group()
    except Exception as e:  # pragma: no cover - reported to the parent
        q.put((rank, False, False, repr(e)))


@pytest.mark.parametrize("world", [2, 3, 4])
def test_two_gloo_ranks_cover_and_reduce(world):
    from zero_sharded_optimizer_flat_gb300 import build_lib
    build_lib.build()
    numel = [1000, 7, 333, 4096, 1, 250]
    bucket = 700
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, numel, bucket, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
    for rank, cover_ok, stats_ok, info in sorted(results):
        assert cover_ok and stats_ok, (rank, info)
    assert len({r[3] for r in results}) == 1  # every rank's shard has the same length
