"""GPU parity of the all-MXFP8 forward (gdpa_fwd_mxfp8: Q, K and V in MXFP8,
the weights P rounded to e4m3 on chip) against the fp64 oracle's MXFP8 path
(every input decoded exactly, exact weights).

The bar is the e4m3-weight bar of tests/parity.py: elementwise
|gpu - oracle| <= 1e-2 + 2U|o| + 2^-4 o_abs (o_abs = the oracle with |V|:
each weight moves by at most half an e4m3 step) and relative L2 <=
2^-4/sqrt(3).  The small batches mix every shape class of the 64-key tile
loop: one key, ragged key tails (1, 31, 33, 63, 65, 127, 129 keys), query
tiles with and without a second tile, an item of two tiles whose second has
one row, sequences with no keys, and enough items per CTA that the scale
words staged ahead cross item boundaries.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from jagged_attention_recommender_gb300 import build as gbuild, gdpa
from jagged_attention_recommender_gb300.workloads import (ACT_SOFTMAX, JaggedBatch, Workload, f32_to_bf16_bits,
                                                          make_batch, offsets_of, to_mx, to_mx_vt)
from tests.parity import assert_parity_mxp, full_output_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    gbuild.build()
    yield


def mxfp8_batch(rng, Lq, Lkv, H, scale):
    Lq, Lkv = np.asarray(Lq), np.asarray(Lkv)
    w = Workload("mxfp8_case", 0, len(Lq), H, 128, ACT_SOFTMAX, 0, scale, "self", mx=True)
    qf = rng.standard_normal((int(Lq.sum()), H, 128)).astype(np.float32)
    kf = rng.standard_normal((int(Lkv.sum()), H, 128)).astype(np.float32)
    vf = rng.standard_normal((int(Lkv.sum()), H, 128)).astype(np.float32)
    b = JaggedBatch(w, f32_to_bf16_bits(qf), f32_to_bf16_bits(kf), f32_to_bf16_bits(vf), offsets_of(Lq),
                    offsets_of(Lkv))
    (b.q8, b.q_sf), (b.k8, b.k_sf) = to_mx(qf), to_mx(kf)
    b.vt8, b.vt_sf = to_mx_vt(vf, b.kv_offsets)
    return b


def run_mxfp8(batch, guard=3, with_lse=False, as_tensor=False):
    w = batch.workload
    H, D, B = w.H, w.D, batch.B
    Tq = int(batch.q_offsets[-1])
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    q8, qs, k8, ks = dev(batch.q8), dev(batch.q_sf), dev(batch.k8), dev(batch.k_sf)
    vt8, vsf = dev(batch.vt8), dev(batch.vt_sf)
    qo, ko = dev(batch.q_offsets), dev(batch.kv_offsets)
    full = torch.full((Tq + 2 * guard, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = full[guard:guard + Tq]
    lse = torch.full((max(Tq, 1), H), float("nan"), dtype=torch.float32, device="cuda") if with_lse else None
    gdpa.gdpa_fwd_mxfp8(q8, qs, k8, ks, vt8, vsf, batch.q_offsets, batch.kv_offsets, qo, ko, B, H, D, w.act,
                        w.scale, out, lse)
    assert gdpa.gdpa_device_status() == gdpa.GDPA_OK
    torch.cuda.synchronize()
    if guard:
        g = torch.cat([full[:guard], full[guard + Tq:]])
        assert torch.isnan(g.float()).all(), "kernel wrote outside its output rows"
    if as_tensor:
        return out
    res = out.float().cpu().numpy().astype(np.float64)
    return (res, lse[:Tq].cpu().numpy().astype(np.float64)) if with_lse else res


def oracle_pair(b):
    """(oracle output, oracle output with |V|) for the batch."""
    w = b.workload
    ref = oracle.gdpa_fwd_mxfp8_batch(b)
    ref_abs = oracle.gdpa_fwd_mxfp8(b.q8, b.q_sf, b.k8, b.k_sf, b.vt8 & 0x7F, b.vt_sf, b.q_offsets, b.kv_offsets,
                                    w.H, w.D, w.act, w.window_blocks, w.scale)
    return ref, ref_abs


def test_mxfp8_self_attention_ragged_tiles():
    rng = np.random.default_rng(5100)
    L = rng.integers(1, 700, size=120, endpoint=True)
    L[:12] = [1, 31, 33, 63, 64, 65, 127, 128, 129, 255, 257, 0]
    b = mxfp8_batch(rng, L, L, 2, 1.0 / np.sqrt(128))
    ref, ref_abs = oracle_pair(b)
    d, rl2 = assert_parity_mxp(run_mxfp8(b), ref, ref_abs, "self")
    print("max |d| %.3e  rel-L2 %.3e" % (d, rl2))


def test_mxfp8_cross_shapes_and_lse():
    rng = np.random.default_rng(5200)
    Lq = np.array([300, 1, 130, 0, 64, 513, 200, 7, 256, 129] * 12)
    Lkv = np.array([5, 900, 0, 3, 128, 129, 1, 257, 65, 2000] * 12)
    b = mxfp8_batch(rng, Lq, Lkv, 4, 1.0 / np.sqrt(128))
    out, lse = run_mxfp8(b, with_lse=True)
    ref, ref_abs = oracle_pair(b)
    assert_parity_mxp(out, ref, ref_abs, "cross")
    # rows without keys: zero output and lse -inf
    qo, ko = b.q_offsets, b.kv_offsets
    for s in np.nonzero(np.diff(ko) == 0)[0]:
        assert np.all(out[qo[s]:qo[s + 1]] == 0) and np.all(lse[qo[s]:qo[s + 1]] == -np.inf)
    assert np.isfinite(lse[np.repeat(np.diff(ko) > 0, np.diff(qo))]).all()


def test_mxfp8_full_workload_every_row():
    batch = make_batch("self_long_mx")
    out = run_mxfp8(batch, guard=0, as_tensor=True)
    w = batch.workload

    def oracle_abs(sub):
        return oracle.gdpa_fwd_mxfp8(sub.q8, sub.q_sf, sub.k8, sub.k_sf, sub.vt8 & 0x7F, sub.vt_sf, sub.q_offsets,
                                     sub.kv_offsets, w.H, w.D, w.act, 0, w.scale)

    worst, rl2, rows = full_output_parity(batch, lambda t0, t1: out[t0:t1].float().cpu().numpy().astype(np.float64),
                                          oracle.gdpa_fwd_mxfp8_batch, "self_long_mx (all MXFP8)",
                                          oracle_abs_fn=oracle_abs)
    print("max |d| %.3e  rel-L2 %.3e  rows %d" % (worst, rl2, rows))


def test_mxfp8_two_calls_in_a_row_agree():
    rng = np.random.default_rng(5300)
    L = rng.integers(1, 900, size=40, endpoint=True)
    b = mxfp8_batch(rng, L, L, 4, 1.0 / np.sqrt(128))
    a1 = run_mxfp8(b, as_tensor=True).clone()
    a2 = run_mxfp8(b, as_tensor=True)
    assert torch.equal(a1, a2)


def test_mxfp8_rejects_bad_arguments():
    qo = np.array([0, 64], np.int32)
    buf = torch.zeros(64 * 128, dtype=torch.uint8, device="cuda")
    sf = torch.full((64 * 4 + 1,), 127, dtype=torch.uint8, device="cuda")
    bf = torch.zeros(64 * 128, dtype=torch.bfloat16, device="cuda")
    for D, act, qs, code in ((64, ACT_SOFTMAX, sf, gdpa.GDPA_ERR_UNSUPPORTED),
                             (128, 1, sf, gdpa.GDPA_ERR_UNSUPPORTED),
                             (128, ACT_SOFTMAX, sf[1:], gdpa.GDPA_ERR_INVALID_ARG)):
        with pytest.raises(gdpa.GdpaError) as e:
            gdpa.gdpa_fwd_mxfp8(buf, qs, buf, sf, buf, sf, qo, qo, 0, 0, 1, 1, D, act, 1.0, bf)
        assert e.value.code == code


def test_mxfp8_device_offsets_past_the_tensors_are_clipped_and_flagged():
    """Device offsets that disagree with the host ones (reaching past the
    tensors): every role clips the item to the rows that exist, nothing is
    written outside `out`, the launch reports GDPA_ERR_INVALID_ARG, and the
    next call with matching offsets is within the bar."""
    rng = np.random.default_rng(5400)
    L = rng.integers(1, 600, size=24, endpoint=True)
    b = mxfp8_batch(rng, L, L, 2, 1.0 / np.sqrt(128))
    w = b.workload
    Tq = int(b.q_offsets[-1])
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    q8, qs, k8, ks, vt8, vsf = (dev(a) for a in (b.q8, b.q_sf, b.k8, b.k_sf, b.vt8, b.vt_sf))
    guard = 5
    full = torch.full((Tq + 2 * guard, w.H, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = full[guard:guard + Tq]
    bad = dev(offsets_of(L * 2 + 7))
    gdpa.gdpa_fwd_mxfp8(q8, qs, k8, ks, vt8, vsf, b.q_offsets, b.kv_offsets, bad, bad, b.B, w.H, w.D, w.act,
                        w.scale, out)
    assert gdpa.gdpa_device_status() == gdpa.GDPA_ERR_INVALID_ARG
    assert torch.isnan(torch.cat([full[:guard], full[guard + Tq:]]).float()).all(), "wrote outside out"
    assert gdpa.gdpa_device_status() == gdpa.GDPA_OK
    qo, ko = dev(b.q_offsets), dev(b.kv_offsets)
    gdpa.gdpa_fwd_mxfp8(q8, qs, k8, ks, vt8, vsf, b.q_offsets, b.kv_offsets, qo, ko, b.B, w.H, w.D, w.act, w.scale,
                        out)
    assert gdpa.gdpa_device_status() == gdpa.GDPA_OK
    ref, ref_abs = oracle_pair(b)
    assert_parity_mxp(out.float().cpu().numpy().astype(np.float64), ref, ref_abs, "after the bad offsets")
