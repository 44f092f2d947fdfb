"""Sharding a jagged batch across ranks (one process per GPU).

Every (sequence, head) of the forward pass is independent, so a batch splits
across ranks by whole sequences with no exchange step: each rank takes a
subset of sequences, rebased to its own offsets, and its outputs are exactly
the rows those sequences would have in the unsharded run.  Sequences are
assigned by longest-processing-time-first over their useful pair counts
(self/cross) so that every rank gets about the same work.

This module holds only index bookkeeping (no attention arithmetic).
"""
from __future__ import annotations

import heapq

import numpy as np

from .metrics import key_count


def sequence_costs(Lq, Lkv, window_blocks: int) -> np.ndarray:
    """Per-sequence cost: useful (query, key) pairs plus one tile of overhead per query tile."""
    Lq = np.asarray(Lq, dtype=np.int64)
    Lkv = np.asarray(Lkv, dtype=np.int64)
    pairs = np.array([key_count(a, b, window_blocks) for a, b in zip(Lq, Lkv)], dtype=np.int64)
    return pairs + 128 * 96 * ((Lq + 127) // 128)


def partition_sequences(Lq, Lkv, world: int, window_blocks: int = 0):
    """LPT partition of sequence indices over ``world`` ranks; each list ascending."""
    if world <= 0:
        raise ValueError("world must be positive")
    cost = sequence_costs(Lq, Lkv, window_blocks)
    order = sorted(range(len(cost)), key=lambda s: (-int(cost[s]), s))
    heap = [(0, r) for r in range(world)]
    parts = [[] for _ in range(world)]
    for s in order:
        load, r = heapq.heappop(heap)
        parts[r].append(s)
        heapq.heappush(heap, (load + int(cost[s]), r))
    return [sorted(p) for p in parts]


def shard(batch, rank: int, world: int):
    """The rank's sub-batch (rebased offsets) and the global sequence ids it holds."""
    Lq, Lkv = batch.lengths()
    seqs = partition_sequences(Lq, Lkv, world, batch.workload.window_blocks)[rank]
    return batch.subset(seqs), seqs


def scatter_rows(global_rows: int, batch, seqs, shard_out: np.ndarray, dest: np.ndarray):
    """Writes a rank's output rows into their places in the unsharded output."""
    qo = batch.q_offsets
    pos = 0
    for s in seqs:
        n = int(qo[s + 1] - qo[s])
        dest[qo[s]:qo[s] + n] = shard_out[pos:pos + n]
        pos += n
    assert pos == shard_out.shape[0] and dest.shape[0] == global_rows
