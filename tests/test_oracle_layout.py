"""Pins for the oracle's flat bucketed layout (deg/zero.py, ZeroMaster __init__/_pieces).

The layout is pinned by brute force: every flat index is mapped forward (bucket -> owning
rank -> shard slot) with plain integer arithmetic written independently of the oracle's
piece walk, and the oracle's shard tables must be exactly the inverse of that map.
"""
import dataclasses

import numpy as np
import pytest

import workloads
from oracle import layout as OL


def forward_map(n_total, bucket, world):
    """Brute force: flat index -> (rank, slot) from the definition, one index at a time."""
    b = max(world, bucket - bucket % world)
    shard_offsets = {}
    out = {}
    for f in range(n_total):
        k = f // b
        s = k * b
        e = min(n_total, s + b)
        L = -(-(e - s) // world) * world
        piece = L // world
        # shard offset of bucket k = sum of earlier pieces
        if k not in shard_offsets:
            shard_offsets[k] = sum(
                (-(-(min(n_total, j * b + b) - j * b) // world) * world) // world for j in range(k))
        q = f - s
        out[f] = (q // piece, shard_offsets[k] + q % piece)
    return out


CASES = [
    ([5], 4, 1), ([5], 4, 2), ([5, 3, 9], 4, 3), ([1, 1, 1, 1, 1, 1, 1], 3, 2),
    ([17, 1, 30, 2, 2], 8, 8), ([100], 7, 8), ([10, 20, 30], 1, 3), ([3], 100, 8),
    ([64, 64, 1, 63], 16, 4), ([2, 3, 5, 7, 11, 13], 5, 3),
]


@pytest.mark.parametrize("numel,bucket,world", CASES)
def test_layout_is_inverse_of_brute_force(numel, bucket, world):
    n = sum(numel)
    fwd = forward_map(n, bucket, world)
    seen = set()
    total = 0
    for r in range(world):
        idx = OL.flat_index_of_shard(numel, bucket, world, r)
        assert idx.shape[0] == OL.shard_len(numel, bucket, world)
        total += idx.shape[0]
        for slot, f in enumerate(idx):
            if f >= 0:
                assert fwd[int(f)] == (r, slot)
                seen.add(int(f))
    # a bijection onto the non-padding slots; the padded total is sum of L
    assert seen == set(range(n))
    assert total == sum(L for _, _, L in OL.buckets(numel, bucket, world))


@pytest.mark.parametrize("numel,bucket,world", CASES)
def test_segments_cover_exactly_the_owned_slots(numel, bucket, world):
    offsets = np.concatenate([[0], np.cumsum(numel)])
    for r in range(world):
        idx = OL.flat_index_of_shard(numel, bucket, world, r)
        covered = np.full(idx.shape[0], -1, dtype=np.int64)
        for i, po, so, ln in OL.segments(numel, bucket, world, r):
            assert ln > 0
            assert np.all(covered[so:so + ln] == -1)
            covered[so:so + ln] = offsets[i] + po + np.arange(ln)
        assert np.array_equal(covered, idx)


def test_bucket_never_below_world():
    assert OL.effective_bucket(3, 8) == 8
    assert OL.effective_bucket(10, 8) == 8
    assert OL.effective_bucket(1 << 25, 8) == 1 << 25
    assert OL.effective_bucket(1 << 25, 3) == (1 << 25) - ((1 << 25) % 3)


def test_workload_shard_lengths():
    """The shard lengths of the four AdamW parameter sets (hand-derived from their shapes)."""
    c1 = workloads.get("c1")
    assert OL.shard_len([p.numel for p in c1.adamw], c1.bucket, 1) == 1_048_832
    c2 = workloads.get("c2")
    n2 = [p.numel for p in c2.adamw]
    assert sum(n2) == 38_652_672
    assert [e - s for s, e, _ in OL.buckets(n2, c2.bucket, 1)] == [33_554_432, 5_098_240]
    c3 = workloads.get("c3")
    assert OL.shard_len([p.numel for p in c3.adamw], c3.bucket, 8) == 8_200_448
    c4 = workloads.get("c4")
    n4 = [p.numel for p in c4.adamw]
    assert sum(n4) == 2_000_000_000
    b4 = OL.buckets(n4, c4.bucket, 8)
    assert len(b4) == 60 and b4[-1][2] == 20_288_512
    assert OL.shard_len(n4, c4.bucket, 8) == 250_000_000


def test_gather_shard_zero_pads():
    numel = [5, 2]
    flat = np.arange(1, 8, dtype=np.float32)
    # bucket 4 (W=2): buckets [0,4) and [4,7) padded to 4; rank 1 owns [2,4) and [6,7)+pad
    sh = OL.gather_shard(flat, numel, 4, 2, 1)
    assert sh.tolist() == [3.0, 4.0, 7.0, 0.0]
    assert OL.decay_mask_of_shard([True, False], numel, 4, 2, 1).tolist() == [1, 1, 0, 0]


@pytest.mark.parametrize("numel,bucket,world", CASES)
def test_sampled_slot_map_equals_enumeration(numel, bucket, world):
    for r in range(world):
        idx = OL.flat_index_of_shard(numel, bucket, world, r)
        slots = np.arange(idx.shape[0])
        assert np.array_equal(OL.flat_index_of_slots(numel, bucket, world, r, slots), idx)
        owner = OL.param_of_flat(numel, idx)
        offsets = np.concatenate([[0], np.cumsum(numel)])
        for f, i in zip(idx, owner):
            if f >= 0:
                assert offsets[i] <= f < offsets[i + 1]


def test_round_robin_muon_ownership_counts():
    """Whole-parameter Muon ownership (bluscript_zero_ckpt.cpp, ShardedMuon: each matrix has one
    owner rank; matrix i belongs to rank i mod W): over the 1.1B Llama-style set's 96 matrices
    and W = 8, every matrix has exactly one owner, every rank owns 12, and rank 0's twelve (six
    matrices per layer, so every eighth one) are Wq, Wv and gate_up, four of each, in model
    order."""
    c3 = workloads.get("c3")
    assert len(c3.muon) == 96
    seen = {}
    for r in range(c3.world):
        w = dataclasses.replace(c3, rank=r)
        own = w.owned_muon()
        assert len(own) == 12
        for p in own:
            assert p.name not in seen
            seen[p.name] = r
    assert len(seen) == 96
    own0 = c3.owned_muon()
    assert [p.shape for p in own0] == [(2048, 2048), (2048, 512), (2048, 11264)] * 4
    assert [p.name for p in own0] == [f"l{4 * q + k}.{n}" for q in range(4) for k, n in
                                      enumerate(("wq", "wv", "gate_up"))]
    assert [c3.muon.index(p) for p in own0] == list(range(0, 96, 8))
