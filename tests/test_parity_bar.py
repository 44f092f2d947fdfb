"""Pins the few-key allowance of the parity bar (tests/parity.py) on the CPU.

A one-key GELU row's exact output is o = gelu(s) v.  Arithmetic that rounds
P = gelu(s) to bf16, multiplies by the bf16 value exactly in fp32 and rounds
the result to bf16 -- the kernel's order of operations -- is correct bf16
arithmetic, so the bar must accept it.  These tests emulate exactly that
with numpy on two million one-key rows drawn like the QK-normed workloads
(s uniform on [-17, 17], v ~ N(0, 1) in bf16) and check that

* the error never exceeds 2U|o| + U^2|o| (U = 2^-8, bf16's unit roundoff):
  the allowance 1e-2 + 2U|o| covers every such row;
* the error comes within a few percent of 2U|o|, and a sizeable share of
  rows exceeds 1.5U|o|: an allowance of 1.5U|o| (P's rounding counted as
  2^-9) would reject correctly rounded results, so 2U is the tight factor.
"""
from __future__ import annotations

import numpy as np
import torch

from jagged_attention_recommender_gb300.workloads import bf16_bits_to_f64, f32_to_bf16_bits
from tests import parity

U = parity.U_BF16


def _one_key_rows(n=2_000_000, seed=0):
    rng = np.random.default_rng(seed)
    s = rng.uniform(-17.0, 17.0, n)
    p = torch.nn.functional.gelu(torch.from_numpy(s), approximate="tanh").numpy()
    v = bf16_bits_to_f64(f32_to_bf16_bits(rng.standard_normal(n).astype(np.float32)))
    exact = p * v
    p_bf16 = bf16_bits_to_f64(f32_to_bf16_bits(p.astype(np.float32)))
    acc = (p_bf16 * v).astype(np.float32)  # exact: 8-bit by 8-bit significands fit fp32
    out = bf16_bits_to_f64(f32_to_bf16_bits(acc))
    return exact, out


def test_unit_roundoff_is_the_half_ulp_of_bf16():
    # 1 + 2^-8 lies half-way between 1 and the next bf16 value 1 + 2^-7: RNE
    # rounds it to 1, an error of exactly U relative to the rounded value
    x = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8], np.float32)
    r = bf16_bits_to_f64(f32_to_bf16_bits(x))
    assert r[0] == 1.0 and r[1] == 1.0 + 2.0 ** -6
    assert abs(r[0] - x[0]) / x[0] <= U


def test_few_key_allowance_covers_correct_bf16_arithmetic():
    exact, out = _one_key_rows()
    d = np.abs(out - exact)
    assert np.all(d <= (2 * U + U * U) * np.abs(exact) + 1e-300)
    assert np.all(d <= parity.bar(exact, few_keys=True))


def test_few_key_allowance_is_tight():
    exact, out = _one_key_rows()
    m = np.abs(exact) > 1e-3
    r = np.abs(out - exact)[m] / np.abs(exact)[m]
    assert r.max() >= 1.9 * U          # the worst rows nearly reach 2U
    assert np.mean(r > 1.5 * U) > 1e-3  # 1.5U would reject thousands of correct rows
    # and with the constant part: rows with |o| large enough that 2U|o| > 1e-2
    big = np.abs(exact) > 8.0
    assert np.any(np.abs(out - exact)[big] > 1e-2 + 1.5 * U * np.abs(exact)[big])


# ---------------------------------------------------------------- e4m3 weights

def _e4m3_weight_rows(n_rows=2000, n_keys=1024, seed=1):
    """Softmax rows with their weights rounded to e4m3 the way the MXFP8
    kernel does: per 32 keys a power-of-two scale 2^e with the block's
    largest weight in (224, 448], codes by torch's float8_e4m3fn conversion,
    the row sum over the unrounded weights.  Scores N(0, 1) (unit-variance
    Q and K at scale 1/sqrt(D)), values N(0, 1)."""
    rng = np.random.default_rng(seed)
    s = rng.standard_normal((n_rows, n_keys))
    v = rng.standard_normal((n_rows, n_keys))
    p = np.exp(s - s.max(axis=1, keepdims=True))
    pb = p.reshape(n_rows, n_keys // 32, 32)
    e = np.ceil(np.log2(pb.max(axis=2)) - np.log2(448.0))
    y = (pb / np.ldexp(1.0, e.astype(np.int64))[..., None]).astype(np.float32)
    q = torch.from_numpy(y).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    pq = (q * np.ldexp(1.0, e.astype(np.int64))[..., None]).reshape(n_rows, n_keys)
    l = p.sum(axis=1)
    exact = (p * v).sum(axis=1) / l
    got = (pq * v).sum(axis=1) / l
    o_abs = (p * np.abs(v)).sum(axis=1) / l
    return exact, got, o_abs, y


def test_e4m3_weight_bar_covers_rounded_weights():
    exact, got, o_abs, y = _e4m3_weight_rows()
    assert y.max() <= 448.0 and y.max() > 224.0  # the scale rule: no code saturates
    d = np.abs(got - exact)
    assert np.all(d <= parity.MXP_REL * o_abs)
    assert parity.rel_l2(got, exact) <= parity.MXP_REL_L2


def test_e4m3_weight_bar_is_tight():
    exact, got, o_abs, _ = _e4m3_weight_rows()
    # the RMS bound is reached to within a factor 2 (the relative step of
    # e4m3 is 2^-3 .. 2^-4 over a binade, so the RMS sits below the bound),
    # and the bf16 bar would reject these correctly rounded results
    rl2 = parity.rel_l2(got, exact)
    assert 0.5 * parity.MXP_REL_L2 <= rl2 <= parity.MXP_REL_L2
    assert rl2 > parity.REL_L2
