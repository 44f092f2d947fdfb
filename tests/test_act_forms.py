"""CPU checks of the two sigma forms the kernels evaluate GELU with
(gelu(x) = x sigma(2u), u = sqrt(2/pi) (x + 0.044715 x^3)), emulated in fp32
with numpy, against torch's exact tanh-GELU in fp64.

The special-function-unit form computes t = -log2(e) s (A + C s^2) with
fp32 products, then 2^t, d = 1 + 2^t and s / d.  Emulated here with
correctly rounded fp32 exp2 and division, it must stay within the bound the
GPU test allows for the hardware instructions (2^-19 |x| + 2^-24): the
roundings of the emulation alone use a small part of it, which leaves room
for the approximate exp2 and reciprocal (about 2^-22 relative each).
"""
from __future__ import annotations

import numpy as np
import torch


LOG2E = np.float32(1.4426950408889634)


def sfu_form_fp32(x: np.ndarray, silu: bool = False) -> np.ndarray:
    """The kernels' SFU sigma route in fp32 (exact exp2 / division stand in for the approximations)."""
    s = x.astype(np.float32)
    A = np.float32(1.0) if silu else np.float32(1.5957691216057308)
    C = np.float32(0.0) if silu else np.float32(A * np.float32(0.044715))
    NA, NC = np.float32(-LOG2E * A), np.float32(-LOG2E * C)
    t = (s * (NC * (s * s) + NA)).astype(np.float32)
    with np.errstate(over="ignore"):
        e = np.exp2(t.astype(np.float64)).astype(np.float32)  # rounded once to fp32 (inf for large t)
        d = (e + np.float32(1.0)).astype(np.float32)
        y = (s * (np.float32(1.0) / d).astype(np.float32)).astype(np.float32)
    return y


def test_sfu_form_within_the_gpu_bound_of_exact_gelu():
    x = np.linspace(-17.0, 17.0, 1 << 18).astype(np.float32)
    y = sfu_form_fp32(x).astype(np.float64)
    ref = torch.nn.functional.gelu(torch.from_numpy(x.astype(np.float64)), approximate="tanh").numpy()
    d = np.abs(y - ref)
    bound = 2.0 ** -19 * np.abs(x.astype(np.float64)) + 2.0 ** -24
    assert (d <= bound).all()
    # the emulation's own roundings use at most half of the bound
    assert (d <= 0.5 * bound + 2.0 ** -25).all()


def test_sfu_form_saturates_and_silu():
    big = np.array([20.0, 40.0, 1e3, -20.0, -40.0, -1e3], np.float32)
    y = sfu_form_fp32(big)
    np.testing.assert_allclose(y, [20.0, 40.0, 1e3, 0.0, 0.0, 0.0], atol=1e-5, rtol=1e-6)
    assert not np.isnan(y).any()
    x = np.linspace(-20.0, 20.0, 4001).astype(np.float32)
    ref = torch.nn.functional.silu(torch.from_numpy(x.astype(np.float64))).numpy()
    assert np.abs(sfu_form_fp32(x, silu=True) - ref).max() <= 1e-5
