"""Work and traffic counts used to report throughput.

Useful FLOPs count only the (query, key) pairs a query really attends over:
4 * D * H per pair (the Q.K^T and P.V contractions, two FLOPs per
multiply-add), activation excluded.  Algorithmic bytes count one bf16 read of
Q, K, V and one bf16 write of O.
"""
from __future__ import annotations

from .workloads import BLOCK, JaggedBatch


def key_count(Lq: int, Lkv: int, window_blocks: int) -> int:
    """Number of (query, key) pairs a sequence attends over (useful pairs)."""
    if window_blocks < 0:  # sliding window of W tokens: query i sees min(i + 1, W) keys
        W, L = -window_blocks, int(Lq)
        m = min(W, L)
        return m * (m + 1) // 2 + (L - m) * W
    if window_blocks == 0:
        return int(Lq) * int(Lkv)
    # own block causal + (window_blocks - 1) full previous blocks, clipped at 0
    total = 0
    L = int(Lq)
    for i0 in range(0, L, BLOCK):
        rows = min(BLOCK, L - i0)
        blk = i0 // BLOCK
        prev = min(blk, window_blocks - 1) * BLOCK
        total += rows * prev + rows * (rows + 1) // 2
    return total


def useful_pairs(batch: JaggedBatch) -> int:
    Lq, Lkv = batch.lengths()
    wb = batch.workload.window_blocks
    return sum(key_count(a, b, wb) for a, b in zip(Lq, Lkv))


def useful_flops(batch: JaggedBatch) -> float:
    """4 * D * H * (unmasked pairs): Q.K^T and P.V, activation excluded."""
    return 4.0 * batch.D * batch.H * useful_pairs(batch)


def algorithmic_bytes(batch: JaggedBatch) -> float:
    """Read Q, K, V once and write O once, bf16 (MXFP8 Q and K: one byte an
    element plus one scale byte per 32)."""
    Tq = int(batch.q_offsets[-1])
    Tkv = int(batch.kv_offsets[-1])
    if batch.workload.mx:
        qk = batch.H * batch.D * (1.0 + 1.0 / 32)
        return qk * (Tq + Tkv) + 2.0 * batch.H * batch.D * (Tq + Tkv)
    return 2.0 * batch.H * batch.D * (2 * Tq + 2 * Tkv)
