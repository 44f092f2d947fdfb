"""Pins of the oracle's MXFP8 path (CPU only).

The MX decode is pinned element by element to torch's own float8 types, and
the MX forward to the (separately pinned) bf16 forward: an e4m3 element
times a power-of-two scale is exactly a bf16 value, so decoding the codes
with torch, rounding to bf16 (checked exact) and running the bf16 oracle must
give the MX oracle's output bit for bit.  Scales that differ per 32-element
block make a wrong block index, a swapped operand or a dropped scale fail.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from jagged_attention_recommender_gb300.workloads import (ACT_GELU_TANH, ACT_SILU, ACT_SOFTMAX,
                                                          f32_to_bf16_bits, offsets_of, to_mx)


def test_e4m3_decode_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_double(c) for c in codes])
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    assert np.isnan(got).sum() == 2  # S.1111.111
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x38] == 1.0


def test_e8m0_decode_matches_torch():
    if not hasattr(torch, "float8_e8m0fnu"):
        pytest.skip("torch without float8_e8m0fnu")
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = np.array([oracle.e8m0_to_double(c) for c in codes])
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])
    assert got[127] == 1.0 and got[128] == 2.0


def _torch_dequant_bf16(codes, sf):
    """MX -> bf16 bits through torch's float8 types (exactness checked)."""
    T, H, D = codes.shape
    x = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32)
    s = torch.pow(torch.tensor(2.0, dtype=torch.float64), torch.from_numpy(sf.astype(np.int64) - 127)).float()
    y = (x.reshape(T, H, D // 32, 32) * s[..., None]).reshape(T, H, D).numpy()
    bits = f32_to_bf16_bits(y)
    back = (bits.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(back, y), "MX value not exact in bf16"
    return bits


def _random_mx(rng, T, H, D):
    """N(0, 1) rows quantised, every block's scale then moved by -2..+2
    (values of order one, scales that differ from block to block), and one
    element in 16 replaced by a code from the whole non-NaN range."""
    codes, sf = to_mx(rng.standard_normal((T, H, D)).astype(np.float32))
    sf = (sf.astype(np.int64) + rng.integers(-2, 2, size=sf.shape, endpoint=True)).astype(np.uint8)
    wild = rng.integers(0, 256, size=codes.shape, dtype=np.uint8)
    wild[(wild & 0x7F) == 0x7F] = 0x38
    pick = rng.random(codes.shape) < 1.0 / 16
    codes = np.where(pick, wild >> 2 | (wild & 0x80), codes).astype(np.uint8)  # wild codes kept below 2^1
    return codes, sf


@pytest.mark.parametrize("act,window,D", [(ACT_SOFTMAX, 0, 128), (ACT_GELU_TANH, 0, 128), (ACT_SILU, 0, 64),
                                          (ACT_SOFTMAX, 2, 128), (ACT_SOFTMAX, -40, 64)])
def test_mx_forward_equals_bf16_forward_on_torch_dequantised_inputs(act, window, D):
    rng = np.random.default_rng(900 + D + 7 * act + window)
    H = 2
    L = np.array([1, 70, 130, 5, 0, 200]) if window == 0 else np.array([1, 70, 130, 5, 200])
    Lkv = np.array([3, 200, 1, 64, 9, 130]) if window == 0 else L
    qo, ko = offsets_of(L), offsets_of(Lkv)
    q8, qs = _random_mx(rng, int(qo[-1]), H, D)
    k8, ks = _random_mx(rng, int(ko[-1]), H, D)
    v = f32_to_bf16_bits(rng.standard_normal((int(ko[-1]), H, D)).astype(np.float32))
    scale = 1.0 / np.sqrt(D) if act == ACT_SOFTMAX else 0.05
    got = oracle.gdpa_fwd_mx(q8, qs, k8, ks, v, qo, ko, H, D, act, window, scale)
    ref = oracle.gdpa_fwd(_torch_dequant_bf16(q8, qs), _torch_dequant_bf16(k8, ks), v, qo, ko, H, D, act, window,
                          scale)
    assert np.array_equal(got, ref)
    # and the scales matter: one block's scale doubled changes exactly the
    # rows that read it
    qs2 = qs.copy()
    qs2[qo[1] + 3, 1, 1] += 1
    got2 = oracle.gdpa_fwd_mx(q8, qs2, k8, ks, v, qo, ko, H, D, act, window, scale)
    changed = np.argwhere(np.any(got2 != got, axis=-1))
    assert [tuple(r) for r in changed] == [(qo[1] + 3, 1)]


def test_mx_forward_rejects_bad_block_size():
    q8 = np.zeros((1, 1, 48), np.uint8)
    sf = np.full((1, 1, 1), 127, np.uint8)
    v = np.zeros((1, 1, 48), np.uint16)
    o = np.array([0, 1], np.int32)
    with pytest.raises(ValueError):
        oracle.gdpa_fwd_mx(q8, sf, q8, sf, v, o, o, 1, 48, ACT_SOFTMAX, 0, 1.0)


def test_to_mx_is_the_ocp_recipe():
    """The input generator's quantiser: block scale 2^(floor(log2 amax) - 8),
    every element within half an e4m3 step of x / scale (clamped to 448)."""
    rng = np.random.default_rng(77)
    x = (rng.standard_normal((50, 3, 64)) * np.exp(rng.uniform(-6, 6, size=(50, 3, 1)))).astype(np.float32)
    x[0, 0, :32] = 0.0
    codes, sf = to_mx(x)
    xb = x.reshape(50, 3, 2, 32).astype(np.float64)
    amax = np.abs(xb).max(-1)
    e = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1))) - 8, 0).astype(np.int64)
    assert np.array_equal(sf.astype(np.int64) - 127, e.astype(np.int64))
    dec = np.vectorize(oracle.e4m3_to_double)(codes).reshape(50, 3, 2, 32) * np.ldexp(1.0, e)[..., None]
    y = np.clip(xb / np.ldexp(1.0, e)[..., None], -448, 448)
    # e4m3 spacing at |y|: 2^(floor(log2|y|) - 3), at least 2^-9 (subnormals)
    ulp = np.ldexp(1.0, np.maximum(np.floor(np.log2(np.maximum(np.abs(y), 2.0 ** -9))) - 3, -9).astype(np.int64))
    assert np.all(np.abs(dec / np.ldexp(1.0, e)[..., None] - y) <= ulp / 2)


def test_mx_forward_closed_form_two_blocks():
    """A hand-built case: D = 64 (two scale blocks), one query, two keys.
    e4m3 codes: 0x38 = 1.0, 0x3C = 1.5, 0x30 = 0.5, 0xB8 = -1.0; E8M0 codes:
    126 = 1/2, 127 = 1, 128 = 2, 129 = 4.
      q  = [2 x32, 0.75 x32]           (1.0 * 2, 1.5 * 1/2)
      k0 = [1 x32, 4 x32]              (1.0 * 1, 1.0 * 4)
      k1 = [0.5 x32, -1 x32]           (0.5 * 1, -1.0 * 1)
    so <q, k0> = 64 + 96 = 160, <q, k1> = 32 - 24 = 8; with scale 1/32 the
    scores are 5 and 1/4, and with v0 = 1, v1 = -2 the softmax output is
    (e^5 - 2 e^(1/4)) / (e^5 + e^(1/4)) in every coordinate."""
    import math

    D = 64
    q8 = np.concatenate([np.full(32, 0x38), np.full(32, 0x3C)]).astype(np.uint8).reshape(1, 1, D)
    qs = np.array([128, 126], np.uint8).reshape(1, 1, 2)
    k8 = np.stack([np.full(D, 0x38), np.concatenate([np.full(32, 0x30), np.full(32, 0xB8)])]).astype(np.uint8)
    k8 = k8.reshape(2, 1, D)
    ks = np.array([[127, 129], [127, 127]], np.uint8).reshape(2, 1, 2)
    v = f32_to_bf16_bits(np.stack([np.full(D, 1.0), np.full(D, -2.0)]).astype(np.float32)).reshape(2, 1, D)
    o = np.array([0, 1], np.int32)
    ko = np.array([0, 2], np.int32)
    got = oracle.gdpa_fwd_mx(q8, qs, k8, ks, v, o, ko, 1, D, ACT_SOFTMAX, 0, 1.0 / 32)
    want = (math.exp(5.0) - 2.0 * math.exp(0.25)) / (math.exp(5.0) + math.exp(0.25))
    assert np.allclose(got, want, rtol=1e-14, atol=0)


# ---------------------------------------------------------------- V in MXFP8 (key-major)

def _torch_vt_to_bf16(vt8, vt_sf, kv_offsets, H, D):
    """Key-major MX V -> bf16 bits ``[Tkv, H, D]`` through torch's float8
    type, read back by the layout's definition (sequence b at column
    32 * sum of its predecessors' block counts; scale row = column // 32)."""
    ko = np.asarray(kv_offsets, dtype=np.int64)
    L = np.diff(ko)
    starts = np.concatenate([[0], np.cumsum(32 * ((L + 31) // 32))])
    x = torch.from_numpy(vt8).view(torch.float8_e4m3fn).to(torch.float64).numpy()  # [H*D, VT]
    s = np.ldexp(1.0, vt_sf.astype(np.int64) - 127)                               # [VT/32, H*D]
    out = np.zeros((int(ko[-1]), H * D))
    for b in range(len(L)):
        cols = starts[b] + np.arange(L[b])
        out[ko[b]:ko[b + 1]] = (x[:, cols] * s[cols // 32, :].T).T
    y = out.astype(np.float32)
    assert np.array_equal(y.astype(np.float64), out), "MX value not exact in float32"
    bits = f32_to_bf16_bits(y)
    back = (bits.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(back, y), "MX value not exact in bf16"
    return bits.reshape(-1, H, D)


def _random_vt(rng, kv_offsets, H, D):
    """V drawn N(0, 1), quantised key-major, then every block's scale moved
    by -2..+2 so that neighbouring blocks (and rows) differ."""
    from jagged_attention_recommender_gb300.workloads import to_mx_vt

    v = rng.standard_normal((int(kv_offsets[-1]), H, D)).astype(np.float32)
    vt8, vsf = to_mx_vt(v, kv_offsets)
    vsf = (vsf.astype(np.int64) + rng.integers(-2, 2, size=vsf.shape, endpoint=True)).astype(np.uint8)
    return v, vt8, vsf


def test_vt_layout_and_quantiser():
    """to_mx_vt places sequence b at column 32 * sum ceil(Lkv / 32), zero
    fills the rest of its last block, takes the OCP block scale of each 32
    keys of a (head, coordinate) row, and each element is within half an
    e4m3 step of v / scale; the oracle counts the same row length."""
    from jagged_attention_recommender_gb300.workloads import to_mx_vt, vt_columns

    rng = np.random.default_rng(31)
    Lkv = np.array([5, 0, 64, 33, 100])
    ko = offsets_of(Lkv)
    H, D = 2, 32
    v = (rng.standard_normal((int(ko[-1]), H, D)) * np.exp(rng.uniform(-4, 4, size=(int(ko[-1]), H, 1))))
    v = v.astype(np.float32)
    vt8, vsf = to_mx_vt(v, ko)
    col = vt_columns(ko)
    assert list(col) == [0, 32, 32, 96, 160, 288]
    assert vt8.shape == (H * D, 288) and vsf.shape == (9, H * D)
    assert oracle.vt_columns(ko) == 288
    for b in range(len(Lkv)):  # padding columns are code 0
        assert not vt8[:, col[b] + Lkv[b]:col[b + 1]].any()
    # per block: scale 2^(floor(log2 amax) - 8) and elements within half a step
    dec = torch.from_numpy(vt8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for b in range(len(Lkv)):
        for c0 in range(0, int(Lkv[b]), 32):
            keys = np.arange(c0, min(c0 + 32, int(Lkv[b])))
            xb = v[ko[b] + keys].reshape(len(keys), H * D).astype(np.float64)  # [keys, rows]
            amax = np.abs(xb).max(0)
            e = np.floor(np.log2(amax)) - 8
            blk = (col[b] + c0) // 32
            assert np.array_equal(vsf[blk].astype(np.int64) - 127, e.astype(np.int64))
            y = np.clip(xb / np.ldexp(1.0, e.astype(np.int64)), -448, 448)
            ulp = np.ldexp(1.0, np.maximum(np.floor(np.log2(np.maximum(np.abs(y), 2.0 ** -9))) - 3, -9).astype(np.int64))
            got = dec[:, col[b] + keys].T
            assert np.all(np.abs(got - y) <= ulp / 2)


@pytest.mark.parametrize("act,window,D", [(ACT_SOFTMAX, 0, 128), (ACT_GELU_TANH, 0, 64), (ACT_SILU, 0, 128),
                                          (ACT_SOFTMAX, 2, 64), (ACT_SOFTMAX, -40, 128)])
def test_mxfp8_forward_equals_mx_forward_on_torch_dequantised_v(act, window, D):
    """All-MXFP8 forward == the (pinned) Q/K-MX forward with V decoded by
    torch into bf16 (exact): bit for bit, over ragged sequences whose key
    counts are not multiples of 32 (and one empty sequence)."""
    rng = np.random.default_rng(1900 + D + 7 * act + window)
    H = 2
    L = np.array([1, 70, 130, 5, 0, 200]) if window == 0 else np.array([1, 70, 130, 5, 200])
    Lkv = np.array([3, 200, 1, 64, 9, 130]) if window == 0 else L
    qo, ko = offsets_of(L), offsets_of(Lkv)
    q8, qs = _random_mx(rng, int(qo[-1]), H, D)
    k8, ks = _random_mx(rng, int(ko[-1]), H, D)
    _, vt8, vsf = _random_vt(rng, ko, H, D)
    scale = 1.0 / np.sqrt(D) if act == ACT_SOFTMAX else 0.05
    got = oracle.gdpa_fwd_mxfp8(q8, qs, k8, ks, vt8, vsf, qo, ko, H, D, act, window, scale)
    ref = oracle.gdpa_fwd_mx(q8, qs, k8, ks, _torch_vt_to_bf16(vt8, vsf, ko, H, D), qo, ko, H, D, act, window,
                             scale)
    assert np.array_equal(got, ref)


def test_mxfp8_v_scale_bump_adds_exactly_that_block():
    """P does not depend on V, so doubling one block of V (its scale code
    + 1) adds the output of that block alone: o(V + dV) - o(V) = o(dV), with
    dV the 32 values of the block; nothing outside (sequence, head,
    coordinate) of the block moves."""
    rng = np.random.default_rng(4242)
    H, D = 2, 64
    L = np.array([40, 90, 70])
    qo = offsets_of(L)
    q8, qs = _random_mx(rng, int(qo[-1]), H, D)
    k8, ks = _random_mx(rng, int(qo[-1]), H, D)
    _, vt8, vsf = _random_vt(rng, qo, H, D)
    scale = 1.0 / 8
    base = oracle.gdpa_fwd_mxfp8(q8, qs, k8, ks, vt8, vsf, qo, qo, H, D, ACT_SOFTMAX, 0, scale)
    b, h, d, blk_in_seq = 1, 1, 37, 2  # keys 64..89 of sequence 1 (the sequence's last, partial block)
    col0 = 32 * ((40 + 31) // 32)
    vsf2 = vsf.copy()
    vsf2[col0 // 32 + blk_in_seq, h * D + d] += 1
    bumped = oracle.gdpa_fwd_mxfp8(q8, qs, k8, ks, vt8, vsf2, qo, qo, H, D, ACT_SOFTMAX, 0, scale)
    vfull = _torch_vt_to_bf16(vt8, vsf, qo, H, D)
    dv = np.zeros_like(vfull)
    keys = qo[b] + 32 * blk_in_seq + np.arange(90 - 64)
    dv[keys, h, d] = vfull[keys, h, d]
    delta = oracle.gdpa_fwd_mx(q8, qs, k8, ks, dv, qo, qo, H, D, ACT_SOFTMAX, 0, scale)
    diff = bumped - base
    assert np.allclose(diff, delta, rtol=1e-12, atol=1e-12)  # fp64 rounding of the two sums
    moved = np.argwhere(diff != 0)
    assert moved.size and set(map(tuple, moved[:, 1:])) == {(h, d)}
    assert moved[:, 0].min() >= qo[b] and moved[:, 0].max() < qo[b + 1]


def test_mxfp8_forward_rejects_a_wrong_row_length():
    H, D = 1, 32
    ko = np.array([0, 5], np.int32)
    q8 = np.full((5, H, D), 0x38, np.uint8)
    sf = np.full((5, H, 1), 127, np.uint8)
    vt8 = np.zeros((H * D, 64), np.uint8)  # the layout's row length is 32
    vsf = np.full((2, H * D), 127, np.uint8)
    with pytest.raises(ValueError):
        oracle.gdpa_fwd_mxfp8(q8, sf, q8, sf, vt8, vsf, ko, ko, H, D, ACT_SOFTMAX, 0, 1.0)
