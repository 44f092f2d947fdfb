"""GPU parity of the MXFP8 forward (gdpa_fwd_mx) against the fp64 oracle's MX
path (e4m3 elements times E8M0 block scales, decoded exactly).

Both sides take the same codes, so the only differences are the kernel's:
fp32 accumulation of exact e4m3 products in the score MMA, bf16 P and the
bf16 output -- the bf16 forward's bar (tests/parity.py), with the few-key
allowance 2U|o| (U = 2^-8) on the small cases: with QK-norm and one key, an
ALU activation's output is act(s) v with |act(s)| up to 16, and the bf16
roundings of P and of the output move it by up to 2U|o|.  The full-size
workload keeps the plain bar and is compared over every row.  Batches are large
enough that every CTA walks several items, so the scale words staged ahead
cross item boundaries.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from jagged_attention_recommender_gb300 import build as gbuild, gdpa
from jagged_attention_recommender_gb300.workloads import (ACT_GELU_TANH, ACT_SILU, ACT_SOFTMAX, Workload,
                                                          JaggedBatch, f32_to_bf16_bits, make_batch, offsets_of,
                                                          to_mx)
from tests.parity import assert_parity as _assert_parity, full_output_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    gbuild.build()
    yield


def mx_batch(rng, Lq, Lkv, H, act, scale, qk_norm=False):
    Lq, Lkv = np.asarray(Lq), np.asarray(Lkv)
    w = Workload("mx_case", 0, len(Lq), H, 128, act, 0, scale, "self", mx=True)
    qf = rng.standard_normal((int(Lq.sum()), H, 128)).astype(np.float32)
    kf = rng.standard_normal((int(Lkv.sum()), H, 128)).astype(np.float32)
    if qk_norm:  # rows of L2 norm 4, as the cross workloads' QK-norm
        qf *= 4.0 / np.linalg.norm(qf, axis=-1, keepdims=True)
        kf *= 4.0 / np.linalg.norm(kf, axis=-1, keepdims=True)
    v = f32_to_bf16_bits(rng.standard_normal((int(Lkv.sum()), H, 128)).astype(np.float32))
    b = JaggedBatch(w, f32_to_bf16_bits(qf), f32_to_bf16_bits(kf), v, offsets_of(Lq), offsets_of(Lkv))
    (b.q8, b.q_sf), (b.k8, b.k_sf) = to_mx(qf), to_mx(kf)
    return b


def run_mx(batch, guard=3, with_lse=False, as_tensor=False):
    w = batch.workload
    H, D, B = w.H, w.D, batch.B
    Tq = int(batch.q_offsets[-1])
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    q8, qs, k8, ks = dev(batch.q8), dev(batch.q_sf), dev(batch.k8), dev(batch.k_sf)
    v = dev(batch.v.view(np.int16)).view(torch.bfloat16)
    qo, ko = dev(batch.q_offsets), dev(batch.kv_offsets)
    full = torch.full((Tq + 2 * guard, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = full[guard:guard + Tq]
    lse = torch.full((max(Tq, 1), H), float("nan"), dtype=torch.float32, device="cuda") if with_lse else None
    gdpa.gdpa_fwd_mx(q8, qs, k8, ks, v, batch.q_offsets, batch.kv_offsets, qo, ko, B, H, D, w.act, w.scale, out, lse)
    assert gdpa.gdpa_device_status() == gdpa.GDPA_OK
    torch.cuda.synchronize()
    if guard:
        g = torch.cat([full[:guard], full[guard + Tq:]])
        assert torch.isnan(g.float()).all(), "kernel wrote outside its output rows"
    if as_tensor:
        return out
    res = out.float().cpu().numpy().astype(np.float64)
    return (res, lse[:Tq].cpu().numpy().astype(np.float64)) if with_lse else res


def assert_parity(got, ref, what):
    return _assert_parity(got, ref, what, few_keys=True)


@pytest.mark.parametrize("act", [ACT_SOFTMAX, ACT_GELU_TANH, ACT_SILU])
def test_mx_self_attention_parity(act):
    rng = np.random.default_rng(3100 + act)
    L = rng.integers(1, 400, size=96, endpoint=True)
    L[:6] = [1, 127, 128, 129, 256, 0]
    scale = 1.0 / np.sqrt(128) if act == ACT_SOFTMAX else 1.0
    b = mx_batch(rng, L, L, 2, act, scale, qk_norm=act != ACT_SOFTMAX)
    assert_parity(run_mx(b), oracle.gdpa_fwd_mx_batch(b), "act %d" % act)


def test_mx_cross_shapes_and_lse():
    rng = np.random.default_rng(3200)
    Lq = np.array([300, 1, 130, 0, 64, 513, 200, 7] * 20)
    Lkv = np.array([5, 900, 0, 3, 128, 129, 1, 257] * 20)
    b = mx_batch(rng, Lq, Lkv, 4, ACT_SOFTMAX, 1.0 / np.sqrt(128))
    out, lse = run_mx(b, with_lse=True)
    assert_parity(out, oracle.gdpa_fwd_mx_batch(b), "cross")
    # lse of the MX scores: the bf16 oracle on the exact dequantised inputs
    # gives the same scores, so its backward's lse is the reference
    deq = lambda c, s: f32_to_bf16_bits(
        (torch.from_numpy(c).view(torch.float8_e4m3fn).float().reshape(*c.shape[:2], 4, 32)
         * torch.pow(2.0, torch.from_numpy(s.astype(np.float32)) - 127)[..., None]).reshape(c.shape).numpy())
    rl = oracle.gdpa_bwd(deq(b.q8, b.q_sf), deq(b.k8, b.k_sf), b.v, np.zeros_like(b.v), b.q_offsets, b.kv_offsets,
                         4, 128, ACT_SOFTMAX, 0, b.workload.scale)[3]
    fin = np.isfinite(rl)
    assert np.array_equal(fin, np.isfinite(lse)) and np.all(lse[~fin] == -np.inf)
    assert np.abs(lse[fin] - rl[fin]).max() <= 2e-3


def test_mx_full_workload_every_row():
    batch = make_batch("self_long_mx")
    out = run_mx(batch, guard=0, as_tensor=True)
    full_output_parity(batch, lambda t0, t1: out[t0:t1].float().cpu().numpy().astype(np.float64),
                       oracle.gdpa_fwd_mx_batch, "self_long_mx")


def test_mx_rejects_bad_arguments():
    qo = np.array([0, 64], np.int32)
    buf = torch.zeros(64 * 128, dtype=torch.uint8, device="cuda")
    sf = torch.full((64 * 4 + 1,), 127, dtype=torch.uint8, device="cuda")
    bf = torch.zeros(64 * 128, dtype=torch.bfloat16, device="cuda")
    for D, qs, code in ((64, sf, gdpa.GDPA_ERR_UNSUPPORTED), (128, sf[1:], gdpa.GDPA_ERR_INVALID_ARG)):
        with pytest.raises(gdpa.GdpaError) as e:
            gdpa.gdpa_fwd_mx(buf, qs, buf, sf, bf, qo, qo, 0, 0, 1, 1, D, ACT_SOFTMAX, 1.0, bf)
        assert e.value.code == code
