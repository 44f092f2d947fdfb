"""Pins of the fp64 backward oracle to things other than itself (CPU only).

* library autograd: torch's float64 autograd through a padded-dense forward
  built from library routines (einsum, masked softmax / tanh-GELU, logsumexp),
  on every shape class: ragged and empty sequences, cross attention, windows;
* finite differences of the oracle's own forward (a different code path) for
  a handful of coordinates;
* closed forms: a single key gives dq = dk = 0 and dv = sum of dO; constant
  values give dq = dk = 0 (softmax); zero upstream gradient gives zeros;
* the GELU derivative against a central difference of the GELU.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from jagged_attention_recommender_gb300.workloads import (
    ACT_GELU_TANH, ACT_SILU, ACT_SOFTMAX, BLOCK, bf16_bits_to_f64)
from tests.helpers import bits, small_batch, with_values


def rand_dout(rng, batch):
    w = batch.workload
    return bits(rng.standard_normal((int(batch.q_offsets[-1]), w.H, w.D)).astype(np.float32))


def torch_grads(batch, dout):
    """Reference gradients by torch autograd, float64, one sequence at a time."""
    w = batch.workload
    qf = torch.tensor(bf16_bits_to_f64(batch.q), requires_grad=True)
    kf = torch.tensor(bf16_bits_to_f64(batch.k), requires_grad=True)
    vf = torch.tensor(bf16_bits_to_f64(batch.v), requires_grad=True)
    do = torch.tensor(bf16_bits_to_f64(dout))
    qo, ko = batch.q_offsets, batch.kv_offsets
    loss = torch.zeros((), dtype=torch.float64)
    lse = torch.zeros((int(qo[-1]), w.H), dtype=torch.float64)
    if w.act == ACT_SOFTMAX:
        lse[:] = -torch.inf
    for b in range(len(qo) - 1):
        Lq, Lkv = int(qo[b + 1] - qo[b]), int(ko[b + 1] - ko[b])
        if Lq == 0 or Lkv == 0:
            continue
        Q = qf[qo[b]:qo[b + 1]].transpose(0, 1)   # [H, Lq, D]
        K = kf[ko[b]:ko[b + 1]].transpose(0, 1)
        V = vf[ko[b]:ko[b + 1]].transpose(0, 1)
        S = w.scale * torch.einsum("hid,hjd->hij", Q, K)
        i = torch.arange(Lq)[:, None]
        j = torch.arange(Lkv)[None, :]
        mask = torch.ones((Lq, Lkv), dtype=torch.bool)
        if w.window_blocks > 0:
            mask = (j <= i) & ((i // BLOCK) - (j // BLOCK) <= w.window_blocks - 1)
        elif w.window_blocks < 0:  # sliding window of W tokens
            mask = (j <= i) & (i - j < -w.window_blocks)
        rows = mask.any(dim=1)
        if w.act == ACT_SOFTMAX:
            Sm = S.masked_fill(~mask, -torch.inf)
            l = torch.logsumexp(Sm, dim=-1)                       # [H, Lq]
            P = torch.exp(Sm - torch.where(rows, l, torch.zeros_like(l))[..., None])
            P = torch.where(rows[:, None], P, torch.zeros_like(P))
            lse[qo[b]:qo[b + 1]] = torch.where(rows, l, torch.full_like(l, -torch.inf)).transpose(0, 1).detach()
        elif w.act == ACT_SILU:
            P = torch.nn.functional.silu(S) * mask / Lkv
        else:
            P = torch.nn.functional.gelu(S, approximate="tanh") * mask / Lkv
        O = torch.einsum("hij,hjd->hid", P, V)
        loss = loss + (O * do[qo[b]:qo[b + 1]].transpose(0, 1)).sum()
    if loss.requires_grad:
        loss.backward()
    z = lambda t: t.grad.numpy() if t.grad is not None else np.zeros(t.shape)
    return z(qf), z(kf), z(vf), lse.numpy()


def oracle_grads(batch, dout):
    return oracle.gdpa_bwd_batch(batch, dout, nthreads=2)


def assert_close(got, ref, what, rtol=1e-9):
    scale = max(1.0, float(np.abs(ref).max(initial=0.0)))
    assert np.allclose(got, ref, rtol=0, atol=rtol * scale), "%s: max |d| %.3e" % (what, np.abs(got - ref).max())


CASES = [
    # (Lq, Lkv, H, D, act, window, qk_norm)
    ([5, 1, 37, 0, 12], [5, 1, 37, 0, 12], 2, 16, ACT_SOFTMAX, 0, False),
    ([40, 3, 70], [7, 0, 19], 3, 8, ACT_SOFTMAX, 0, False),
    ([40, 3, 70], [7, 1, 19], 2, 16, ACT_GELU_TANH, 0, True),
    ([130, 64, 65], [130, 64, 65], 1, 8, ACT_SOFTMAX, 2, False),   # windows, partial blocks
    ([0, 9], [4, 0], 2, 8, ACT_GELU_TANH, 0, True),                 # all rows empty
    ([40, 3, 70], [7, 1, 19], 2, 16, ACT_SILU, 0, True),              # SiLU cross
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_oracle_bwd_matches_torch_autograd(case):
    Lq, Lkv, H, D, act, wb, qkn = CASES[case]
    rng = np.random.default_rng(800 + case)
    b = small_batch(rng, Lq, Lkv, H, D, act=act, window_blocks=wb, qk_norm=qkn, scale=1.0 if act else None)
    do = rand_dout(rng, b)
    dq, dk, dv, lse = oracle_grads(b, do)
    rq, rk, rv, rl = torch_grads(b, do)
    assert_close(dq, rq, "dq")
    assert_close(dk, rk, "dk")
    assert_close(dv, rv, "dv")
    fin = np.isfinite(rl)
    assert np.array_equal(fin, np.isfinite(lse)), "lse: empty-row pattern"
    assert np.allclose(lse[fin], rl[fin], rtol=0, atol=1e-12)


@pytest.mark.parametrize("act", [ACT_SOFTMAX, ACT_GELU_TANH, ACT_SILU])
def test_oracle_bwd_matches_finite_differences_of_forward(act):
    # d/dx of L = sum(dO * O) by central differences of the forward oracle,
    # perturbing one bf16 input to its neighbours (exact bf16 values)
    rng = np.random.default_rng(900 + act)
    b = small_batch(rng, [6, 3], [5, 4], 1, 8, act=act, qk_norm=bool(act), scale=1.0 if act else None)
    do = rand_dout(rng, b)
    dof = bf16_bits_to_f64(do)
    dq, dk, dv, _ = oracle_grads(b, do)

    def loss(bb):
        return float((oracle.gdpa_fwd_batch(bb, nthreads=1) * dof).sum())

    for name, grad in (("q", dq), ("k", dk), ("v", dv)):
        arr = getattr(b, name)
        for idx in [(0, 0, 0), (2, 0, 5), (len(arr) - 1, 0, 7)]:
            up, dn = arr.copy(), arr.copy()
            up[idx] = arr[idx] + 1   # next bf16 value (same sign and exponent range here)
            dn[idx] = arr[idx] - 1
            xu = bf16_bits_to_f64(up)[idx]
            xd = bf16_bits_to_f64(dn)[idx]
            fd = (loss(with_values(b, **{name: up})) - loss(with_values(b, **{name: dn}))) / (xu - xd)
            # one bf16 step is ~2^-8 relative: the central difference is exact to second order
            tol = 5e-3 * max(1.0, abs(grad[idx]))
            assert abs(fd - grad[idx]) <= tol, (name, idx, fd, grad[idx])


def test_single_key_softmax_closed_form():
    rng = np.random.default_rng(910)
    b = small_batch(rng, [7, 4], [1, 1], 2, 8)
    do = rand_dout(rng, b)
    dq, dk, dv, lse = oracle_grads(b, do)
    assert np.all(dq == 0) and np.allclose(dk, 0, atol=1e-15)
    dof = bf16_bits_to_f64(do)
    assert np.allclose(dv[0], dof[0:7].sum(axis=0), atol=1e-12)
    assert np.allclose(dv[1], dof[7:11].sum(axis=0), atol=1e-12)
    # lse of one key is its score
    qf, kf = bf16_bits_to_f64(b.q), bf16_bits_to_f64(b.k)
    s = b.workload.scale * np.einsum("thd,hd->th", qf[0:7], kf[0])
    assert np.allclose(lse[0:7], s, atol=1e-12)


def test_constant_values_give_zero_query_and_key_gradients():
    rng = np.random.default_rng(911)
    b = small_batch(rng, [9, 33], [12, 20], 2, 16)
    v = np.broadcast_to(b.v[:1], b.v.shape).copy()
    b = with_values(b, v=v)
    dq, dk, dv, _ = oracle_grads(b, rand_dout(rng, b))
    assert np.abs(dq).max() < 1e-12 and np.abs(dk).max() < 1e-12


def test_zero_upstream_gradient():
    rng = np.random.default_rng(912)
    b = small_batch(rng, [9, 33], [12, 20], 2, 16, act=ACT_GELU_TANH, qk_norm=True, scale=1.0)
    do = np.zeros_like(b.q)
    dq, dk, dv, _ = oracle_grads(b, do)
    assert not dq.any() and not dk.any() and not dv.any()


def test_gelu_grad_matches_central_difference():
    for x in np.linspace(-8, 8, 97):
        h = 1e-5
        fd = (oracle.gelu_tanh(x + h) - oracle.gelu_tanh(x - h)) / (2 * h)
        assert abs(oracle.gelu_tanh_grad(x) - fd) < 1e-8


def test_silu_and_its_grad_closed_forms():
    # silu(0) = 0, silu'(0) = 1/2; silu(x) -> x and silu'(x) -> 1 for large x;
    # silu(-x) = silu(x) - x; central difference of the oracle's silu
    assert oracle.silu(0.0) == 0.0 and oracle.silu_grad(0.0) == 0.5
    assert abs(oracle.silu(40.0) - 40.0) < 1e-12 and abs(oracle.silu_grad(40.0) - 1.0) < 1e-12
    for x in np.linspace(-8, 8, 65):
        assert abs(oracle.silu(-x) - (oracle.silu(x) - x)) < 1e-12
        fd = (oracle.silu(x + 1e-5) - oracle.silu(x - 1e-5)) / 2e-5
        assert abs(oracle.silu_grad(x) - fd) < 1e-8
