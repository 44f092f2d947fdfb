"""Seeded synthetic jagged GDPA workloads.

This module only draws inputs: sequence lengths, bf16 value tensors laid out
``[tokens, H, D]`` and int32 offset prefix sums.  It holds none of the
attention arithmetic, so the CUDA path and the CPU oracle can both be fed from
it without sharing any of the method.

The five workloads follow the shape classes the GEM training write-up lists
for its attention variants (techfeed summary of "GEM Training", section
"why LLM infrastructure does not carry over": jagged user histories of
hundreds to tens of thousands of tokens; self-attention, long-query/short-KV
cross attention, short-query/long-KV pooled attention), plus the 64-token
block-aligned window of the "BlockAttention" section.  Exact sizes and
distributions are the benchmark configurations of this project:

==============  ====================================================================
name            recipe
==============  ====================================================================
tiny            B=4, H=2, D=64, L ~ U{1..128}; softmax; scale 1/sqrt(D)
self_long       B=256, H=4, D=128, L = clip(round(lognormal(6.9, 0.8)), 100, 4096)
cross_gelu      B=512, H=4, D=128, Lq ~ U{256..4096}, Lkv ~ U{8..64}; Q, K rows
                L2-normalised per (token, head) then x4; GELU; scale 1.0
pma             B=256, H=8, D=64, 32 seed queries shared by every sample
                (materialised per sample), Lkv = clip(round(lognormal(7.6, 1.0)),
                100, 16384); softmax; scale 1/sqrt(D)
block_window    B=64, H=4, D=128, L = 64 * U{8..512}; window of 4 blocks of 64
                (own block causal + 3 previous); softmax; scale 1/sqrt(D)
sliding_window  B=64, H=4, D=128, L ~ U{512..32768}; causal sliding window of
                256 tokens (window_blocks = -256); softmax; scale 1/sqrt(D)
cross_silu      cross_gelu's shapes and QK-norm with SiLU instead of GELU
pffn            B=256, H=4, D=128, Lq ~ U{256..4096}, Lkv = 512: a per-sample FFN
                gelu(x W1^T) W2 as GDPA (K = W1, V = W2, 512 hidden units per
                sample); GELU; scale 1/sqrt(D); no QK-norm
self_long_mx    self_long's lengths and values with Q and K in MXFP8: e4m3
                elements, one E8M0 scale per 32 coordinates (OCP MX recipe:
                scale 2^(floor(log2 amax) - 8), elements rounded to nearest
                even and clamped to +-448); V bf16
==============  ====================================================================

Draw order (fixed): lengths first, then one 63-bit sub-seed per value tensor
(Q, K, V), all from ``numpy.random.default_rng(seed)``.  Values are drawn in
fixed chunks of tokens, each chunk from ``default_rng([sub_seed, chunk])``, so
the result does not depend on how many threads draw it.  Values are float32
N(0, 1), rounded to bf16 with round-to-nearest-even and kept as raw uint16
bit patterns.
"""
from __future__ import annotations

import dataclasses
import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

ACT_SOFTMAX = 0
ACT_GELU_TANH = 1
ACT_SILU = 2

CHUNK_TOKENS = 16384


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    B: int
    H: int
    D: int
    act: int
    window_blocks: int
    scale: float
    kind: str  # "self", "cross", "pma", "window", "ffn"
    mx: bool = False  # Q and K also drawn as MXFP8 (e4m3 codes + E8M0 block scales)


WORKLOADS = {
    "tiny": Workload("tiny", 0, 4, 2, 64, ACT_SOFTMAX, 0, 1.0 / math.sqrt(64), "self"),
    "self_long": Workload("self_long", 1, 256, 4, 128, ACT_SOFTMAX, 0, 1.0 / math.sqrt(128), "self"),
    "cross_gelu": Workload("cross_gelu", 2, 512, 4, 128, ACT_GELU_TANH, 0, 1.0, "cross"),
    "pma": Workload("pma", 3, 256, 8, 64, ACT_SOFTMAX, 0, 1.0 / math.sqrt(64), "pma"),
    "block_window": Workload("block_window", 4, 64, 4, 128, ACT_SOFTMAX, 4, 1.0 / math.sqrt(128), "window"),
    "cross_silu": Workload("cross_silu", 6, 512, 4, 128, ACT_SILU, 0, 1.0, "cross"),
    "pffn": Workload("pffn", 7, 256, 4, 128, ACT_GELU_TANH, 0, 1.0 / math.sqrt(128), "ffn"),
    # window_blocks < 0: a causal sliding window of -window_blocks tokens
    "sliding_window": Workload("sliding_window", 5, 64, 4, 128, ACT_SOFTMAX, -256, 1.0 / math.sqrt(128), "window"),
    "self_long_mx": Workload("self_long_mx", 1, 256, 4, 128, ACT_SOFTMAX, 0, 1.0 / math.sqrt(128), "self", mx=True),
}

MX_BLOCK = 32

PMA_SEEDS = 32
BLOCK = 64


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (round to nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def _mx_blocks(xb: np.ndarray):
    """OCP MX quantisation of float32 blocks ``[..., 32]``: returns (e4m3
    codes uint8 ``[..., 32]``, E8M0 scale codes uint8 ``[...]``).  The block
    scale is 2^(floor(log2 amax) - 8) (8 = the largest e4m3 exponent),
    elements are x / scale clamped to +-448 and rounded to nearest even by
    torch's float8_e4m3fn conversion; an all-zero block takes scale 1."""
    import torch

    xb = np.ascontiguousarray(xb, dtype=np.float32)
    amax = np.abs(xb).max(axis=-1)
    _, ex = np.frexp(amax)  # amax = m 2^ex, m in [0.5, 1): floor(log2 amax) = ex - 1
    e = np.where(amax > 0, ex - 1 - 8, 0).clip(-127, 127).astype(np.int32)
    sf = (e + 127).astype(np.uint8)
    y = np.clip(xb * np.ldexp(np.float32(1.0), -e)[..., None].astype(np.float32), -448.0, 448.0)
    codes = torch.from_numpy(np.ascontiguousarray(y)).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes.numpy(), sf


def to_mx(x: np.ndarray):
    """OCP MX quantisation of float32 ``[T, H, D]`` rows in blocks of 32
    coordinates: returns (e4m3 codes uint8 ``[T, H, D]``, E8M0 scale codes
    uint8 ``[T, H, D // 32]``), each block as :func:`_mx_blocks`."""
    T, H, D = x.shape
    codes, sf = _mx_blocks(np.asarray(x, dtype=np.float32).reshape(T, H, D // MX_BLOCK, MX_BLOCK))
    return codes.reshape(T, H, D), sf


def vt_columns(kv_offsets) -> np.ndarray:
    """First column of each sequence in the key-major MXFP8 layout of V:
    ``P_b = 32 * sum_{b' < b} ceil(Lkv_b' / 32)`` (int64 ``[B+1]``, last
    entry = VT, the row length)."""
    L = np.diff(np.asarray(kv_offsets, dtype=np.int64))
    col = np.zeros(len(L) + 1, dtype=np.int64)
    col[1:] = np.cumsum(MX_BLOCK * ((L + MX_BLOCK - 1) // MX_BLOCK))
    return col


def to_mx_vt(v: np.ndarray, kv_offsets):
    """V ``[Tkv, H, D]`` (float32) in MXFP8 along the keys: returns (codes
    uint8 ``[H*D, VT]``, scales uint8 ``[VT // 32, H*D]``).  Row h*D + d holds
    coordinate d of head h; sequence b's keys sit at columns
    ``[P_b, P_b + Lkv_b)`` (:func:`vt_columns`), the rest of its last block is
    zero; scale ``[c, h*D + d]`` covers columns ``[32 c, 32 c + 32)`` of that
    row; blocks as :func:`_mx_blocks`."""
    Tkv, H, D = v.shape
    ko = np.asarray(kv_offsets, dtype=np.int64)
    col = vt_columns(ko)
    VT = int(col[-1])
    vt8 = np.zeros((H * D, VT), dtype=np.uint8)
    vsf = np.full((VT // MX_BLOCK, H * D), 127, dtype=np.uint8)
    for b in range(len(ko) - 1):
        L = int(ko[b + 1] - ko[b])
        if L == 0:
            continue
        n = (L + MX_BLOCK - 1) // MX_BLOCK
        x = np.zeros((n * MX_BLOCK, H * D), dtype=np.float32)
        x[:L] = np.asarray(v[ko[b]:ko[b + 1]], dtype=np.float32).reshape(L, H * D)
        codes, sf = _mx_blocks(x.reshape(n, MX_BLOCK, H * D).transpose(0, 2, 1))  # [n, H*D, 32], [n, H*D]
        c0 = int(col[b])
        vt8[:, c0:c0 + n * MX_BLOCK] = codes.transpose(1, 0, 2).reshape(H * D, n * MX_BLOCK)
        vsf[c0 // MX_BLOCK:c0 // MX_BLOCK + n] = sf
    return vt8, vsf


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b).astype(np.uint32) << 16).view(np.float32)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def draw_lengths(w: Workload, rng: np.random.Generator, B: int | None = None):
    """Per-sequence (Lq, Lkv) for ``B`` sequences (default: the workload's B)."""
    B = w.B if B is None else B
    if w.name == "tiny":
        L = rng.integers(1, 128, size=B, endpoint=True)
        return L, L
    if w.name in ("self_long", "self_long_mx"):
        L = np.clip(np.round(rng.lognormal(6.9, 0.8, size=B)), 100, 4096).astype(np.int64)
        return L, L
    if w.name in ("cross_gelu", "cross_silu"):
        Lq = rng.integers(256, 4096, size=B, endpoint=True)
        Lkv = rng.integers(8, 64, size=B, endpoint=True)
        return Lq, Lkv
    if w.name == "pma":
        Lkv = np.clip(np.round(rng.lognormal(7.6, 1.0, size=B)), 100, 16384).astype(np.int64)
        return np.full(B, PMA_SEEDS, dtype=np.int64), Lkv
    if w.name == "block_window":
        L = BLOCK * rng.integers(8, 512, size=B, endpoint=True)
        return L, L
    if w.name == "sliding_window":
        L = rng.integers(512, 32768, size=B, endpoint=True)
        return L, L
    if w.name == "pffn":
        return rng.integers(256, 4096, size=B, endpoint=True), np.full(B, 512, dtype=np.int64)
    raise KeyError(w.name)


def offsets_of(lengths) -> np.ndarray:
    c = np.cumsum(np.asarray(lengths, dtype=np.int64))
    if c.size and c[-1] >= 2**31:
        raise ValueError("total token count does not fit int32 offsets")
    off = np.zeros(len(lengths) + 1, dtype=np.int32)
    off[1:] = c
    return off


def _normal_chunked(sub_seed: int, tokens: int, H: int, D: int, threads: int) -> np.ndarray:
    out = np.empty((tokens, H, D), dtype=np.float32)
    n_chunks = (tokens + CHUNK_TOKENS - 1) // CHUNK_TOKENS

    def fill(c):
        lo = c * CHUNK_TOKENS
        hi = min(tokens, lo + CHUNK_TOKENS)
        g = np.random.default_rng([sub_seed, c])
        out[lo:hi] = g.standard_normal((hi - lo, H, D), dtype=np.float32)

    if threads > 1 and n_chunks > 1:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(fill, range(n_chunks)))
    else:
        for c in range(n_chunks):
            fill(c)
    return out


def _qk_norm_x4(x: np.ndarray) -> np.ndarray:
    """Input recipe of the cross workload: each (token, head) row scaled to L2 norm 4."""
    n = np.sqrt(np.einsum("thd,thd->th", x, x, dtype=np.float32))
    return x * (np.float32(4.0) / np.maximum(n, np.float32(1e-30)))[..., None]


@dataclasses.dataclass
class JaggedBatch:
    workload: Workload
    q: np.ndarray          # uint16 bf16 bits [Tq, H, D]
    k: np.ndarray          # uint16 bf16 bits [Tkv, H, D]
    v: np.ndarray          # uint16 bf16 bits [Tkv, H, D]
    q_offsets: np.ndarray  # int32 [B+1]
    kv_offsets: np.ndarray  # int32 [B+1]
    # MXFP8 workloads: e4m3 codes [T, H, D] and E8M0 scales [T, H, D/32] of
    # Q and K (q, k then hold the unquantised values, rounded to bf16)
    q8: np.ndarray | None = None
    q_sf: np.ndarray | None = None
    k8: np.ndarray | None = None
    k_sf: np.ndarray | None = None
    # and V in MXFP8 along the keys (to_mx_vt of the bf16 values of v)
    vt8: np.ndarray | None = None
    vt_sf: np.ndarray | None = None

    @property
    def B(self) -> int:
        return len(self.q_offsets) - 1

    @property
    def H(self) -> int:
        return self.workload.H

    @property
    def D(self) -> int:
        return self.workload.D

    def lengths(self):
        return np.diff(self.q_offsets).astype(np.int64), np.diff(self.kv_offsets).astype(np.int64)

    def subset(self, seqs) -> "JaggedBatch":
        """The batch made of sequences ``seqs`` (in that order), copied contiguous."""
        seqs = [int(s) for s in seqs]
        qo, ko = self.q_offsets, self.kv_offsets
        q = np.concatenate([self.q[qo[s]:qo[s + 1]] for s in seqs]) if seqs else self.q[:0]
        k = np.concatenate([self.k[ko[s]:ko[s + 1]] for s in seqs]) if seqs else self.k[:0]
        v = np.concatenate([self.v[ko[s]:ko[s + 1]] for s in seqs]) if seqs else self.v[:0]

        def rows(a, off):
            if a is None:
                return None
            return np.ascontiguousarray(np.concatenate([a[off[s]:off[s + 1]] for s in seqs]) if seqs else a[:0])

        sub = JaggedBatch(self.workload, np.ascontiguousarray(q), np.ascontiguousarray(k),
                          np.ascontiguousarray(v),
                          offsets_of([qo[s + 1] - qo[s] for s in seqs]),
                          offsets_of([ko[s + 1] - ko[s] for s in seqs]),
                          rows(self.q8, qo), rows(self.q_sf, qo), rows(self.k8, ko), rows(self.k_sf, ko))
        if self.vt8 is not None:
            sub.vt8, sub.vt_sf = to_mx_vt(bf16_bits_to_f32(sub.v), sub.kv_offsets)
        return sub


def make_batch(name: str, B: int | None = None, seed: int | None = None,
               lengths=None, threads: int | None = None) -> JaggedBatch:
    """Draw the seeded batch of workload ``name``.

    ``B`` and ``seed`` override the workload's batch size and seed (smaller
    cases with the same distributions); ``lengths`` = (Lq, Lkv) arrays override
    the length draw entirely (edge-case tests).
    """
    w = WORKLOADS[name]
    seed = w.seed if seed is None else seed
    threads = threads or min(16, os.cpu_count() or 1)
    rng = np.random.default_rng(seed)
    if lengths is None:
        Lq, Lkv = draw_lengths(w, rng, B)
    else:
        Lq, Lkv = (np.asarray(x, dtype=np.int64) for x in lengths)
    subs = [int(s) for s in rng.integers(0, 2**63 - 1, size=3)]
    H, D = w.H, w.D
    Tq, Tkv = int(Lq.sum()), int(Lkv.sum())
    if w.kind == "pma":
        seeds = _normal_chunked(subs[0], PMA_SEEDS, H, D, 1)
        qf = np.empty((Tq, H, D), dtype=np.float32)
        qo = offsets_of(Lq)
        for b in range(len(Lq)):
            n = int(Lq[b])
            qf[qo[b]:qo[b] + n] = seeds[:n]
    else:
        qf = _normal_chunked(subs[0], Tq, H, D, threads)
    kf = _normal_chunked(subs[1], Tkv, H, D, threads)
    if w.kind == "cross":
        qf = _qk_norm_x4(qf)
        kf = _qk_norm_x4(kf)
    mx = (to_mx(qf), to_mx(kf)) if w.mx else None
    q = f32_to_bf16_bits(qf)
    del qf
    k = f32_to_bf16_bits(kf)
    del kf
    v = f32_to_bf16_bits(_normal_chunked(subs[2], Tkv, H, D, threads))
    b = JaggedBatch(w, q, k, v, offsets_of(Lq), offsets_of(Lkv))
    if mx is not None:
        (b.q8, b.q_sf), (b.k8, b.k_sf) = mx
        b.vt8, b.vt_sf = to_mx_vt(bf16_bits_to_f32(v), b.kv_offsets)
    return b
