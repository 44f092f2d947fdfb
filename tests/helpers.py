"""Shared test helpers: small input builders and the padded-dense brute force.

The brute force is deliberately built differently from the oracle: it pads
every sequence to the batch maximum, forms the full [B, H, Lq_max, Lkv_max]
score tensor with one einsum, builds an explicit boolean mask, and takes the
GELU from torch's library routine.  The window mask uses the equivalent
"j <= i and block distance <= W-1" form instead of the oracle's case split.
"""
from __future__ import annotations

import numpy as np
import torch

from jagged_attention_recommender_gb300.workloads import (
    BLOCK, JaggedBatch, Workload, bf16_bits_to_f64, f32_to_bf16_bits, offsets_of)


def bits(x) -> np.ndarray:
    return f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def small_batch(rng, Lq, Lkv, H, D, act=0, window_blocks=0, scale=None, name="custom",
                qk_norm=False) -> JaggedBatch:
    Lq = np.asarray(Lq, dtype=np.int64)
    Lkv = np.asarray(Lkv, dtype=np.int64)
    scale = float(np.float32(1.0 / np.sqrt(D))) if scale is None else float(np.float32(scale))
    q = rng.standard_normal((int(Lq.sum()), H, D)).astype(np.float32)
    k = rng.standard_normal((int(Lkv.sum()), H, D)).astype(np.float32)
    v = rng.standard_normal((int(Lkv.sum()), H, D)).astype(np.float32)
    if qk_norm:
        q = 4 * q / np.linalg.norm(q, axis=-1, keepdims=True)
        k = 4 * k / np.linalg.norm(k, axis=-1, keepdims=True)
    kind = "window" if window_blocks != 0 else "self"
    w = Workload(name, 0, len(Lq), H, D, act, window_blocks, scale, kind)
    return JaggedBatch(w, bits(q), bits(k), bits(v), offsets_of(Lq), offsets_of(Lkv))


def with_values(batch: JaggedBatch, q=None, k=None, v=None, act=None, window_blocks=None,
                scale=None) -> JaggedBatch:
    w = batch.workload
    w2 = Workload(w.name, w.seed, w.B, w.H, w.D, w.act if act is None else act,
                  w.window_blocks if window_blocks is None else window_blocks,
                  w.scale if scale is None else float(np.float32(scale)), w.kind)
    return JaggedBatch(w2, batch.q if q is None else q, batch.k if k is None else k,
                       batch.v if v is None else v, batch.q_offsets, batch.kv_offsets)


def padded_dense(batch: JaggedBatch, causal_only=False) -> np.ndarray:
    """Brute-force reference, fp64 [Tq, H, D]."""
    w = batch.workload
    H, D = w.H, w.D
    qo, ko = batch.q_offsets, batch.kv_offsets
    B = len(qo) - 1
    Lq = np.diff(qo)
    Lkv = np.diff(ko)
    Mq = max(1, int(Lq.max(initial=0)))
    Mk = max(1, int(Lkv.max(initial=0)))
    Q = np.zeros((B, Mq, H, D))
    K = np.zeros((B, Mk, H, D))
    V = np.zeros((B, Mk, H, D))
    qf, kf, vf = bf16_bits_to_f64(batch.q), bf16_bits_to_f64(batch.k), bf16_bits_to_f64(batch.v)
    for b in range(B):
        Q[b, :Lq[b]] = qf[qo[b]:qo[b + 1]]
        K[b, :Lkv[b]] = kf[ko[b]:ko[b + 1]]
        V[b, :Lkv[b]] = vf[ko[b]:ko[b + 1]]
    S = w.scale * np.einsum("bihd,bjhd->bhij", Q, K)
    i = np.arange(Mq)[:, None]
    j = np.arange(Mk)[None, :]
    mask = np.zeros((B, 1, Mq, Mk), dtype=bool)
    for b in range(B):
        m = (i < Lq[b]) & (j < Lkv[b])
        if causal_only:
            m &= j <= i
        elif w.window_blocks > 0:
            m &= (j <= i) & ((i // BLOCK) - (j // BLOCK) <= w.window_blocks - 1)
        elif w.window_blocks < 0:  # sliding window of W tokens: a band of W diagonals
            W = -w.window_blocks
            m &= np.tril(np.ones((Mq, Mk), dtype=bool)) & np.triu(np.ones((Mq, Mk), dtype=bool), -(W - 1))
        mask[b, 0] = m
    if w.act == 0:
        Sm = np.where(mask, S, -np.inf)
        mx = Sm.max(axis=-1, keepdims=True)
        mx = np.where(np.isfinite(mx), mx, 0.0)
        E = np.where(mask, np.exp(Sm - mx), 0.0)
        den = E.sum(axis=-1, keepdims=True)
        O = np.einsum("bhij,bjhd->bihd", E, V)
        den_t = np.transpose(den, (0, 2, 1, 3))  # [B, Mq, H, 1]
        O = np.where(den_t > 0, O / np.where(den_t > 0, den_t, 1.0), 0.0)
    else:
        if w.act == 2:  # SiLU
            G = torch.nn.functional.silu(torch.from_numpy(S)).numpy()
        else:
            G = torch.nn.functional.gelu(torch.from_numpy(S), approximate="tanh").numpy()
        G = np.where(mask, G, 0.0)
        O = np.einsum("bhij,bjhd->bihd", G, V)
        div = np.where(Lkv > 0, Lkv, 1).astype(np.float64)
        O = O / div[:, None, None, None]
        O[Lkv == 0] = 0.0
    out = np.zeros((int(qo[-1]), H, D))
    for b in range(B):
        out[qo[b]:qo[b + 1]] = O[b, :Lq[b]]
    return out


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))
