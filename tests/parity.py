"""The parity bar every GPU test of a forward output uses, in one place.

Workload bar (the target the library is held to): max |gpu - oracle| <= 1e-2
and relative L2 error <= 5e-3, the GPU output in bf16, the oracle in fp64 on
the same bf16 inputs.

Few-key allowance.  The kernel rounds P to bf16 before P.V and rounds the
output to bf16.  bf16 keeps 8 significant bits and rounds to nearest even,
so each rounding moves a value by at most U = 2^-8 of itself (half an ulp,
and an ulp is at most 2^-7 of the value).  A row whose output comes from one
key -- or from keys whose terms share a sign -- carries both roundings on
its whole value: |gpu - exact| <= (2U + U^2)|o| plus fp32 accumulation and
the ALU activation's own error (both below 1e-6 relative).  With QK-normed
scores up to 16 and one key, |o| = |act(s) v| reaches ~50, where 2U|o| is
~0.4 -- far above 1e-2 -- for results that are correctly rounded bf16
arithmetic.  So rows of the few-key cases (one-key GELU/SiLU rows, the first
rows of a sliding window, MXFP8's one-key rows) are held to

    |gpu - oracle| <= 1e-2 + 2U |oracle|,   U = 2^-8

elementwise.  ``tests/test_parity_bar.py`` pins this on the CPU: correctly
rounded bf16 arithmetic of one-key rows comes within a few percent of 2U|o|
(so no tighter factor is safe), and never exceeds it.  The five workloads of
the target keep the plain bar; their full-size outputs are compared with the
oracle over every row (``full_output_parity``).

MXFP8 weights (gdpa_fwd_mxfp8).  There the kernel also rounds each weight
P_ij to e4m3 (3 mantissa bits) under a per-32-key power-of-two scale that
keeps every code normal or saturation-free, so each weight moves by at most
half an e4m3 step: |dP| <= 2^-4 P (and far less for the few codes left
subnormal).  Summed over the keys with |v_j|, the output moves by at most
2^-4 o_abs, o_abs_i = sum_j P_ij |v_j| / sum_j P_ij (the oracle with |V|),
so the elementwise bar adds that term; and a rounding error uniform on
+-half a step has RMS at most 2^-4 / sqrt(3) of the weight, which bounds the
relative L2 error when V's signs are random:

    |gpu - oracle| <= 1e-2 + 2U |oracle| + 2^-4 o_abs,   rel-L2 <= 2^-4 / sqrt(3)

``tests/test_parity_bar.py`` pins both on the CPU with e4m3-rounded weights.
"""
from __future__ import annotations

import math

import numpy as np

MAX_ABS = 1e-2
REL_L2 = 5e-3
U_BF16 = 2.0 ** -8  # unit roundoff of bf16 (round to nearest even, 8 significant bits)
FEW_KEY_REL = 2.0 * U_BF16  # P rounded to bf16, then the output rounded to bf16


MXP_REL = 2.0 ** -4              # half an e4m3 step, relative
MXP_REL_L2 = MXP_REL / math.sqrt(3.0)  # RMS of a relative error uniform on +-MXP_REL


def bar(ref: np.ndarray, few_keys: bool = False, ref_abs: np.ndarray | None = None) -> np.ndarray:
    """Elementwise allowance for |gpu - oracle| (``ref_abs``: the oracle with
    |V|, for outputs whose weights were rounded to e4m3)."""
    if ref_abs is not None:
        return MAX_ABS + FEW_KEY_REL * np.abs(ref) + MXP_REL * np.asarray(ref_abs)
    if few_keys:
        return MAX_ABS + FEW_KEY_REL * np.abs(ref)
    return np.full(ref.shape, MAX_ABS)


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


def assert_parity(got, ref, what: str = "", few_keys: bool = False):
    """Asserts the bar elementwise and rel-L2 over the whole array; returns (max |d|, rel-L2)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, "%s: shape %s vs %s" % (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), "non-finite output " + what
    if not got.size:
        return 0.0, 0.0
    d = np.abs(got - ref)
    b = bar(ref, few_keys)
    worst = np.unravel_index(np.argmax(d - b), d.shape)
    assert np.all(d <= b), "%s: |d| %.3e > bar %.3e at %s (|ref| %.3g)" % (
        what, d[worst], b[worst], worst, abs(ref[worst]))
    rl2 = rel_l2(got, ref)
    assert rl2 <= REL_L2, "%s: rel L2 %.3e" % (what, rl2)
    return float(d.max()), rl2


def sequence_groups(q_offsets, max_rows: int = 1 << 16, min_seqs: int = 8):
    """Consecutive groups of whole sequences, ~max_rows query rows each (at
    least min_seqs sequences, so the oracle's threads over (sequence, head)
    stay busy)."""
    qo = np.asarray(q_offsets)
    B = len(qo) - 1
    groups, start = [], 0
    while start < B:
        end = start + 1
        while end < B and (qo[end] - qo[start] < max_rows or end - start < min_seqs):
            end += 1
        groups.append(list(range(start, end)))
        start = end
    return groups


def assert_parity_mxp(got, ref, ref_abs, what: str = ""):
    """The e4m3-weight bar (module docstring); returns (max |d|, rel-L2)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, "%s: shape %s vs %s" % (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), "non-finite output " + what
    if not got.size:
        return 0.0, 0.0
    d = np.abs(got - ref)
    b = bar(ref, ref_abs=ref_abs)
    worst = np.unravel_index(np.argmax(d - b), d.shape)
    assert np.all(d <= b), "%s: |d| %.3e > bar %.3e at %s (|ref| %.3g)" % (
        what, d[worst], b[worst], worst, abs(ref[worst]))
    rl2 = rel_l2(got, ref)
    assert rl2 <= MXP_REL_L2, "%s: rel L2 %.3e" % (what, rl2)
    return float(d.max()), rl2


def full_output_parity(batch, got_fn, oracle_fn, what: str = "", few_keys: bool = False,
                       max_rows: int = 1 << 16, oracle_abs_fn=None):
    """Compares every row of a launch's output with the oracle, group by group.

    ``got_fn(t0, t1)`` returns the GPU output rows [t0, t1) as fp64 and
    ``oracle_fn(sub_batch)`` the oracle over a subset of whole sequences; the
    elementwise bar holds in every group and rel-L2 over the whole output.
    With ``oracle_abs_fn`` (the oracle with |V| over a subset) the bar is the
    e4m3-weight one.  Returns (max |d|, rel-L2, rows compared).
    """
    qo = np.asarray(batch.q_offsets)
    num = den = 0.0
    worst = 0.0
    rows = 0
    for seqs in sequence_groups(qo, max_rows):
        t0, t1 = int(qo[seqs[0]]), int(qo[seqs[-1] + 1])
        if t1 == t0:
            continue
        got = np.asarray(got_fn(t0, t1), dtype=np.float64)
        ref = oracle_fn(batch.subset(seqs))
        assert got.shape == ref.shape
        assert np.isfinite(got).all(), "non-finite output %s rows %d..%d" % (what, t0, t1)
        d = np.abs(got - ref)
        b = bar(ref, few_keys, None if oracle_abs_fn is None else oracle_abs_fn(batch.subset(seqs)))
        if not np.all(d <= b):
            i = np.unravel_index(np.argmax(d - b), d.shape)
            raise AssertionError("%s: |d| %.3e > bar %.3e at row %d (|ref| %.3g)" % (
                what, d[i], b[i], t0 + i[0], abs(ref[i])))
        worst = max(worst, float(d.max()))
        num += float(np.sum((got - ref) ** 2))
        den += float(np.sum(ref ** 2))
        rows += t1 - t0
    rl2 = float(np.sqrt(num / den)) if den > 0 else 0.0
    assert rl2 <= (REL_L2 if oracle_abs_fn is None else MXP_REL_L2), "%s: rel L2 %.3e over the whole output" % (
        what, rl2)
    assert rows == int(qo[-1]), "%s: compared %d of %d rows" % (what, rows, int(qo[-1]))
    return worst, rl2, rows
