"""Flat bucketed shard layout — oracle (test infrastructure only).

Source: deg/zero.py, ZeroMaster — class docstring ("laid end to end in a flat vector of N
elements cut into buckets ... the last one padded to a multiple of world. Rank r owns the
r-th of world equal pieces of every bucket; its shard is those pieces concatenated"),
``__init__`` (bucket rounding and the (start, end, padded length) triples) and
``_segments`` / ``_pieces``.
"""
from __future__ import annotations

import bisect

import numpy as np


def effective_bucket(bucket: int, world: int) -> int:
    """Bucket size rounded down to a multiple of ``world`` but never below ``world``
    (ZeroMaster.__init__)."""
    return max(world, bucket - bucket % world)


def buckets(numel: list, bucket: int, world: int) -> list:
    """(start, end, padded length) for every bucket of the flat vector (ZeroMaster.__init__)."""
    n = int(sum(numel))
    b = effective_bucket(bucket, world)
    out = []
    for s in range(0, n, b):
        e = min(n, s + b)
        padded = -(-(e - s) // world) * world  # ceil((e - s) / world) * world
        out.append((s, e, padded))
    return out


def shard_len(numel: list, bucket: int, world: int) -> int:
    return sum(L // world for _, _, L in buckets(numel, bucket, world))


def pieces(numel: list, bucket: int, world: int) -> list:
    """(bucket start, end, padded length, piece length, shard offset) (ZeroMaster._pieces)."""
    out, o = [], 0
    for s, e, L in buckets(numel, bucket, world):
        piece = L // world
        out.append((s, e, L, piece, o))
        o += piece
    return out


def flat_index_of_shard(numel: list, bucket: int, world: int, rank: int) -> np.ndarray:
    """For every slot of rank ``rank``'s shard, the flat index it holds, or -1 for padding.

    Written as the definition reads: walk the buckets, take the rank's piece of each."""
    out = []
    for s, e, L, piece, _ in pieces(numel, bucket, world):
        for j in range(piece):
            f = s + rank * piece + j
            out.append(f if f < e else -1)
    return np.asarray(out, dtype=np.int64)


def segments(numel: list, bucket: int, world: int, rank: int) -> list:
    """(param index, offset in param, shard offset, length) runs covering the rank's shard
    (ZeroMaster._segments over each piece's flat range)."""
    offsets = [0]
    for n in numel:
        offsets.append(offsets[-1] + int(n))
    out = []
    for s, e, L, piece, o in pieces(numel, bucket, world):
        a0 = s + rank * piece
        b0 = min(e, a0 + piece)
        if a0 >= b0:
            continue
        i = bisect.bisect_right(offsets, a0) - 1
        while i < len(numel) and offsets[i] < b0:
            a = max(a0, offsets[i])
            b = min(b0, offsets[i + 1])
            if b > a:
                out.append((i, a - offsets[i], o + (a - a0), b - a))
            i += 1
    return out


def gather_shard(flat: np.ndarray, numel: list, bucket: int, world: int, rank: int, idx=None) -> np.ndarray:
    """Rank ``rank``'s shard of a flat vector, zeros in the padding (ZeroMaster._bucket_values
    then the rank's piece). ``idx`` may pass a precomputed slot -> flat index map."""
    if idx is None:
        idx = flat_index_of_slots(numel, bucket, world, rank, np.arange(shard_len(numel, bucket, world)))
    out = np.zeros(idx.shape[0], dtype=flat.dtype)
    ok = idx >= 0
    out[ok] = flat[idx[ok]]
    return out


def decay_mask_of_shard(decay: list, numel: list, bucket: int, world: int, rank: int) -> np.ndarray:
    """Per shard slot: 1 where the owning parameter takes weight decay, 0 for excluded
    parameters and padding."""
    flat = np.concatenate([np.full(int(n), 1 if d else 0, dtype=np.uint8) for n, d in zip(numel, decay)]) \
        if numel else np.zeros(0, np.uint8)
    return gather_shard(flat, numel, bucket, world, rank)


def flat_index_of_slots(numel: list, bucket: int, world: int, rank: int, slots: np.ndarray) -> np.ndarray:
    """The flat index held by each of the given shard slots (-1 for padding), for sampled
    checks of shards too large to enumerate: find the slot's bucket from the pieces' shard
    offsets, then offset into the rank's piece of that bucket."""
    ps = pieces(numel, bucket, world)
    starts = np.array([p[0] for p in ps], dtype=np.int64)
    ends = np.array([p[1] for p in ps], dtype=np.int64)
    piece = np.array([p[3] for p in ps], dtype=np.int64)
    offs = np.array([p[4] for p in ps], dtype=np.int64)
    slots = np.asarray(slots, dtype=np.int64)
    k = np.searchsorted(offs, slots, side="right") - 1
    f = starts[k] + rank * piece[k] + (slots - offs[k])
    return np.where(f < ends[k], f, -1)


def param_of_flat(numel: list, flat: np.ndarray) -> np.ndarray:
    """Index of the parameter that holds each flat index (-1 stays -1)."""
    offsets = np.concatenate([[0], np.cumsum(np.asarray(numel, dtype=np.int64))])
    flat = np.asarray(flat, dtype=np.int64)
    i = np.searchsorted(offsets, flat, side="right") - 1
    return np.where(flat >= 0, i, -1)
