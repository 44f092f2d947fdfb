"""Pins of the fp64 oracle to things other than itself (CPU only).

* brute force: padded dense attention with explicit masks (tests/helpers.py)
  on tiny inputs of every shape class, including ragged and empty sequences
  and windows with a trailing partial block;
* closed forms: one key, identical keys, constant values, zero scale, GELU
  against torch's tanh-GELU, softmax of two scores = logistic function;
* invariants: sequence permutation, key permutation, head independence,
  linearity in V, per-row score shift, full window = causal attention;
* golden: hand-derived cases stored under tests/golden/.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from jagged_attention_recommender_gb300.workloads import (
    ACT_GELU_TANH, ACT_SOFTMAX, bf16_bits_to_f64, make_batch, offsets_of)
from tests.helpers import bits, padded_dense, small_batch, with_values

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def run(batch, nthreads=2):
    return oracle.gdpa_fwd_batch(batch, nthreads=nthreads)


# ---------------------------------------------------------------- brute force

BRUTE_CASES = [
    # (Lq, Lkv, H, D, act, window, qk_norm)
    ([5, 1, 37, 0, 12], [5, 1, 37, 0, 12], 2, 16, ACT_SOFTMAX, 0, False),
    ([40, 3, 70], [7, 0, 19], 3, 8, ACT_SOFTMAX, 0, False),           # cross, empty KV
    ([40, 3, 70], [7, 1, 19], 2, 16, ACT_GELU_TANH, 0, True),         # GELU cross
    ([40, 3, 70], [7, 0, 19], 2, 16, 2, 0, True),                     # SiLU cross, empty KV
    ([0, 9, 33], [4, 0, 33], 2, 8, ACT_GELU_TANH, 0, True),           # empty Q and empty KV
    ([32, 32], [150, 7], 2, 8, ACT_SOFTMAX, 0, False),                # PMA-like
    ([200, 64, 130], [200, 64, 130], 1, 8, ACT_SOFTMAX, 4, False),    # window, partial tail block
    ([200, 129], [200, 129], 2, 8, ACT_SOFTMAX, 2, False),
    ([190], [190], 1, 8, ACT_SOFTMAX, 1, False),                      # own block only
]


@pytest.mark.parametrize("case", range(len(BRUTE_CASES)))
def test_oracle_matches_padded_dense(case):
    Lq, Lkv, H, D, act, wb, qkn = BRUTE_CASES[case]
    rng = np.random.default_rng(100 + case)
    b = small_batch(rng, Lq, Lkv, H, D, act=act, window_blocks=wb, qk_norm=qkn,
                    scale=1.0 if qkn else None)
    got = run(b)
    ref = padded_dense(b)
    assert got.shape == ref.shape
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-12)


def test_tiny_workload_matches_padded_dense():
    b = make_batch("tiny")
    np.testing.assert_allclose(run(b), padded_dense(b), rtol=1e-11, atol=1e-12)


def test_full_window_is_causal_attention():
    rng = np.random.default_rng(7)
    L = [150, 90]
    b = small_batch(rng, L, L, 2, 8, window_blocks=10)  # 10 blocks > 3 blocks in any sequence
    np.testing.assert_allclose(run(b), padded_dense(b, causal_only=True), rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("W", [1, 2, 63, 64, 65, 130])
def test_sliding_window_matches_padded_dense(W):
    rng = np.random.default_rng(30 + W)
    L = [150, 1, 64, 65, 0, 129]
    b = small_batch(rng, L, L, 2, 8, window_blocks=-W)
    np.testing.assert_allclose(run(b), padded_dense(b), rtol=1e-11, atol=1e-12)


def test_sliding_window_of_one_token_returns_own_value():
    rng = np.random.default_rng(40)
    L = [7, 33]
    b = small_batch(rng, L, L, 2, 8, window_blocks=-1)
    np.testing.assert_array_equal(run(b), bf16_bits_to_f64(b.v))


def test_wide_sliding_window_is_causal_attention():
    rng = np.random.default_rng(41)
    L = [150, 90]
    b = small_batch(rng, L, L, 2, 8, window_blocks=-150)
    np.testing.assert_allclose(run(b), padded_dense(b, causal_only=True), rtol=1e-11, atol=1e-12)


def test_sliding_window_backward_matches_torch_autograd():
    from tests.test_oracle_bwd_pins import assert_close, rand_dout, torch_grads
    rng = np.random.default_rng(42)
    L = [130, 64, 65, 1]
    b = small_batch(rng, L, L, 1, 8, window_blocks=-40)
    do = rand_dout(rng, b)
    dq, dk, dv, lse = oracle.gdpa_bwd_batch(b, do, nthreads=2)
    rq, rk, rv, rl = torch_grads(b, do)
    assert_close(dq, rq, "dq")
    assert_close(dk, rk, "dk")
    assert_close(dv, rv, "dv")
    assert np.allclose(lse, rl, atol=1e-12)


# ---------------------------------------------------------------- closed forms

def test_single_key_softmax_returns_v0_exactly():
    rng = np.random.default_rng(1)
    b = small_batch(rng, [17, 3], [1, 1], 2, 16)
    out = run(b)
    v = bf16_bits_to_f64(b.v)
    assert np.array_equal(out[:17], np.broadcast_to(v[0], (17, 2, 16)))
    assert np.array_equal(out[17:], np.broadcast_to(v[1], (3, 2, 16)))


def test_single_key_gelu_is_gelu_of_score_times_v0():
    rng = np.random.default_rng(2)
    b = small_batch(rng, [11], [1], 3, 16, act=ACT_GELU_TANH, qk_norm=True, scale=1.0)
    out = run(b)
    q, k, v = (bf16_bits_to_f64(x) for x in (b.q, b.k, b.v))
    s = np.einsum("ihd,hd->ih", q, k[0])
    g = torch.nn.functional.gelu(torch.from_numpy(s), approximate="tanh").numpy()
    np.testing.assert_allclose(out, g[..., None] * v[0][None], rtol=1e-12, atol=1e-13)


def test_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(3)
    b = small_batch(rng, [9, 20], [13, 40], 2, 8)
    k = b.k.copy()
    k[:13] = k[0]
    k[13:] = k[13]
    out = run(with_values(b, k=k))
    v = bf16_bits_to_f64(b.v)
    np.testing.assert_allclose(out[:9], np.broadcast_to(v[:13].mean(0), (9, 2, 8)), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(out[9:], np.broadcast_to(v[13:].mean(0), (20, 2, 8)), rtol=1e-12, atol=1e-14)


def test_identical_keys_window_gives_mean_over_window():
    rng = np.random.default_rng(4)
    L = 200
    b = small_batch(rng, [L], [L], 1, 8, window_blocks=2)
    k = b.k.copy()
    k[:] = k[0]
    out = run(with_values(b, k=k))
    v = bf16_bits_to_f64(b.v)[:, 0]
    for i in (0, 1, 63, 64, 65, 127, 128, 150, 199):
        lo = max(0, (i // 64 - 1) * 64)
        np.testing.assert_allclose(out[i, 0], v[lo:i + 1].mean(0), rtol=1e-12, atol=1e-14)


def test_constant_values_give_that_constant():
    rng = np.random.default_rng(5)
    b = small_batch(rng, [30, 5], [44, 9], 2, 8)
    v = bits(np.full(b.v.shape, 0.375))
    out = run(with_values(b, v=v))
    np.testing.assert_allclose(out, 0.375, rtol=1e-14, atol=0)


def test_zero_scale():
    rng = np.random.default_rng(6)
    b = small_batch(rng, [12, 7], [21, 3], 2, 8)
    out = run(with_values(b, scale=0.0))
    v = bf16_bits_to_f64(b.v)
    np.testing.assert_allclose(out[:12], np.broadcast_to(v[:21].mean(0), (12, 2, 8)), rtol=1e-12, atol=1e-14)
    out_g = run(with_values(b, scale=0.0, act=ACT_GELU_TANH))
    assert np.all(out_g == 0.0)


def test_gelu_matches_torch_tanh_gelu():
    xs = np.linspace(-17.0, 17.0, 2001)
    ours = np.array([oracle.gelu_tanh(x) for x in xs])
    ref = torch.nn.functional.gelu(torch.from_numpy(xs), approximate="tanh").numpy()
    np.testing.assert_allclose(ours, ref, rtol=1e-14, atol=1e-15)
    # and it is the tanh form, not the erf form: they differ by up to ~5e-4 near |x| ~ 2.5
    erf = torch.nn.functional.gelu(torch.from_numpy(xs)).numpy()
    assert 1e-4 < np.abs(ours - erf).max() < 1e-3


def test_gelu_large_scores_saturate():
    # gelu(x) -> x for large positive x: o = s * v / Lkv with one key
    rng = np.random.default_rng(8)
    b = small_batch(rng, [4], [1], 1, 4, act=ACT_GELU_TANH, scale=1.0)
    q = bits(np.full(b.q.shape, 4.0))
    k = bits(np.full(b.k.shape, 2.0))  # s = 4 * 2 * 4 = 32
    out = run(with_values(b, q=q, k=k))
    v = bf16_bits_to_f64(b.v)
    np.testing.assert_allclose(out, 32.0 * np.broadcast_to(v[0], out.shape), rtol=1e-15)


# ---------------------------------------------------------------- invariants

def test_sequence_permutation_permutes_outputs():
    rng = np.random.default_rng(9)
    b = small_batch(rng, [10, 50, 3, 27], [12, 8, 30, 1], 2, 8)
    out = run(b)
    perm = [2, 0, 3, 1]
    sub = b.subset(perm)
    out_p = run(sub)
    qo = b.q_offsets
    expect = np.concatenate([out[qo[s]:qo[s + 1]] for s in perm])
    assert np.array_equal(out_p, expect)


@pytest.mark.parametrize("act", [ACT_SOFTMAX, ACT_GELU_TANH])
def test_key_permutation_leaves_outputs(act):
    rng = np.random.default_rng(10)
    b = small_batch(rng, [16, 9], [33, 20], 2, 8, act=act)
    out = run(b)
    perm = np.concatenate([rng.permutation(33), 33 + rng.permutation(20)])
    out_p = run(with_values(b, k=b.k[perm], v=b.v[perm]))
    np.testing.assert_allclose(out_p, out, rtol=1e-12, atol=1e-14)


def test_heads_are_independent():
    rng = np.random.default_rng(11)
    b = small_batch(rng, [21, 6], [21, 6], 3, 8)
    out = run(b)
    k = b.k.copy()
    k[:, 1] = bits(rng.standard_normal(k[:, 1].shape))
    out2 = run(with_values(b, k=k))
    assert np.array_equal(out2[:, 0], out[:, 0]) and np.array_equal(out2[:, 2], out[:, 2])
    assert not np.allclose(out2[:, 1], out[:, 1])


@pytest.mark.parametrize("act", [ACT_SOFTMAX, ACT_GELU_TANH])
def test_linear_in_values(act):
    # small integers keep 2*v1 - v2 exact in bf16
    rng = np.random.default_rng(12)
    b = small_batch(rng, [14, 31], [19, 5], 2, 8, act=act)
    v1 = rng.integers(-4, 5, size=b.v.shape).astype(np.float32)
    v2 = rng.integers(-4, 5, size=b.v.shape).astype(np.float32)
    o1 = run(with_values(b, v=bits(v1)))
    o2 = run(with_values(b, v=bits(v2)))
    o3 = run(with_values(b, v=bits(2 * v1 - v2)))
    np.testing.assert_allclose(o3, 2 * o1 - o2, rtol=1e-10, atol=1e-12)


def test_softmax_invariant_to_per_row_score_shift():
    # k_j + u for one fixed vector u adds q_i.u to every score of row i
    rng = np.random.default_rng(13)
    H, D = 1, 8
    q = rng.integers(-2, 3, size=(6, H, D)).astype(np.float32)
    k = rng.integers(-2, 3, size=(10, H, D)).astype(np.float32)
    u = rng.integers(-3, 4, size=(D,)).astype(np.float32)
    b = small_batch(rng, [6], [10], H, D, scale=0.25)
    b = with_values(b, q=bits(q), k=bits(k))
    o1 = run(b)
    o2 = run(with_values(b, k=bits(k + u)))
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- edge cases

def test_empty_batch_and_all_empty_sequences():
    rng = np.random.default_rng(14)
    b = small_batch(rng, [0, 0], [5, 0], 2, 8)
    assert run(b).shape == (0, 2, 8)
    b2 = small_batch(rng, [7], [0], 2, 8)
    assert np.all(run(b2) == 0.0)


def test_bad_arguments_are_rejected():
    z = np.zeros((4, 1, 8), dtype=np.uint16)
    with pytest.raises(ValueError):  # non-monotone offsets
        oracle.gdpa_fwd(z, z, z, np.array([0, 3, 2], np.int32), np.array([0, 1, 2], np.int32), 1, 8, 0, 0, 1.0)
    with pytest.raises(ValueError):  # window with Lq != Lkv
        oracle.gdpa_fwd(z, z, z, np.array([0, 4], np.int32), np.array([0, 3], np.int32), 1, 8, 0, 2, 1.0)


# ---------------------------------------------------------------- golden

def test_golden_hand_cases():
    with open(os.path.join(GOLDEN, "hand_cases.json")) as f:
        cases = json.load(f)["cases"]
    assert cases
    for c in cases:
        H, D = c["H"], c["D"]
        q = bits(np.array(c["q"], dtype=np.float32).reshape(-1, H, D))
        k = bits(np.array(c["k"], dtype=np.float32).reshape(-1, H, D))
        v = bits(np.array(c["v"], dtype=np.float32).reshape(-1, H, D))
        out = oracle.gdpa_fwd(q, k, v, np.array(c["q_offsets"], np.int32), np.array(c["kv_offsets"], np.int32),
                              H, D, c["act"], c["window_blocks"], c["scale"])
        rows = c.get("rows")
        got = out[rows] if rows is not None else out
        np.testing.assert_allclose(got.reshape(-1), np.array(c["out"], dtype=np.float64), rtol=1e-12,
                                   atol=1e-14, err_msg=c["name"])


@pytest.mark.parametrize("act", [ACT_GELU_TANH, 2])
def test_pffn_is_gdpa_with_weights_as_keys_and_values(act):
    # A per-sample FFN, act(x W1^T) W2 (W1, W2: [hidden, D]), is GDPA with
    # K = W1, V = W2 and the ALU activation: o = (1/hidden) act(x W1^T) W2.
    # Brute force with torch's activation on plain matrices, per sample.
    rng = np.random.default_rng(60 + act)
    Lq, hidden = np.array([5, 17, 1]), np.array([24, 24, 24])
    b = small_batch(rng, Lq, hidden, 1, 16, act=act, scale=0.25)
    got = run(b)
    qf, kf, vf = bf16_bits_to_f64(b.q), bf16_bits_to_f64(b.k), bf16_bits_to_f64(b.v)
    f = (lambda z: torch.nn.functional.gelu(z, approximate="tanh")) if act == ACT_GELU_TANH else torch.nn.functional.silu
    for i in range(len(Lq)):
        x = torch.from_numpy(qf[b.q_offsets[i]:b.q_offsets[i + 1], 0])
        W1 = torch.from_numpy(kf[b.kv_offsets[i]:b.kv_offsets[i + 1], 0])
        W2 = torch.from_numpy(vf[b.kv_offsets[i]:b.kv_offsets[i + 1], 0])
        ffn = (f(0.25 * x @ W1.T) @ W2).numpy()
        np.testing.assert_allclose(got[b.q_offsets[i]:b.q_offsets[i + 1], 0] * hidden[i], ffn, rtol=1e-11, atol=1e-11)
