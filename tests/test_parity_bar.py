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
