"""GPU parity of the causal sliding window (gdpa_fwd_sliding) against the
fp64 oracle (window_blocks = -W in the oracle: keys i - W < j <= i).

The forward workloads' bar (tests/parity.py) with the few-key allowance:
the first rows of a sequence see only a handful of keys, so |o| reaches
|v| ~ 4, and the bf16 roundings of P and of the output move such a row by
up to 2U|o| (U = 2^-8), more than 1e-2 once |o| > 1.3.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from jagged_attention_recommender_gb300 import build as gbuild, gdpa
from jagged_attention_recommender_gb300.workloads import ACT_GELU_TANH, ACT_SOFTMAX, make_batch
from tests.helpers import small_batch
from tests.parity import assert_parity as _assert_parity, full_output_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    gbuild.build()
    yield


def dev(bits_arr):
    return torch.from_numpy(np.ascontiguousarray(bits_arr).view(np.int16)).view(torch.bfloat16).cuda()


def run_sliding(batch, W, guard=3, with_lse=False, as_tensor=False):
    w = batch.workload
    H, D, B = w.H, w.D, len(batch.q_offsets) - 1
    Tq = int(batch.q_offsets[-1])
    q, k, v = dev(batch.q), dev(batch.k), dev(batch.v)
    qo = torch.from_numpy(batch.q_offsets).cuda()
    ko = torch.from_numpy(batch.kv_offsets).cuda()
    full = torch.full((Tq + 2 * guard, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = full[guard:guard + Tq]
    lse = torch.full((Tq, H), float("nan"), dtype=torch.float32, device="cuda") if with_lse else None
    gdpa.gdpa_fwd_sliding(q, k, v, batch.q_offsets, batch.kv_offsets, qo, ko, B, H, D, w.act, W, w.scale, out, lse)
    assert gdpa.gdpa_device_status() == gdpa.GDPA_OK
    torch.cuda.synchronize()
    if guard:
        g = torch.cat([full[:guard], full[guard + Tq:]])
        assert torch.isnan(g.float()).all(), "kernel wrote outside its output rows"
    if as_tensor:
        return out
    res = out.float().cpu().numpy().astype(np.float64)
    if with_lse:
        return res, lse.cpu().numpy().astype(np.float64)
    return res


def assert_parity(got, ref, what):
    return _assert_parity(got, ref, what, few_keys=True)


LENGTHS = [1, 64, 65, 200, 640, 1000, 257, 256]


@pytest.mark.parametrize("W", [1, 17, 64, 65, 200, 1000])
def test_sliding_window_parity(W):
    rng = np.random.default_rng(8000 + W)
    L = np.array(LENGTHS)
    b = small_batch(rng, L, L, 2, 128, window_blocks=-W)
    assert_parity(run_sliding(b, W), oracle.gdpa_fwd_batch(b), "W=%d" % W)


def test_sliding_window_d64_and_lse():
    rng = np.random.default_rng(8100)
    L = np.array([300, 129, 512, 3])
    b = small_batch(rng, L, L, 4, 64, window_blocks=-100)
    out, lse = run_sliding(b, 100, with_lse=True)
    assert_parity(out, oracle.gdpa_fwd_batch(b), "D=64")
    rl = oracle.gdpa_bwd_batch(b, np.zeros_like(b.q))[3]
    assert np.abs(lse - rl).max() <= 2e-3


def test_sliding_window_full_workload_every_row():
    batch = make_batch("sliding_window")
    w = batch.workload
    out = run_sliding(batch, -w.window_blocks, guard=0, as_tensor=True)
    full_output_parity(batch, lambda t0, t1: out[t0:t1].float().cpu().numpy().astype(np.float64),
                       oracle.gdpa_fwd_batch, "sliding_window", few_keys=True)


def test_sliding_window_rejects_bad_arguments():
    qo = np.array([0, 64], np.int32)
    for act, W, ko, code in ((ACT_GELU_TANH, 8, qo, gdpa.GDPA_ERR_UNSUPPORTED),
                             (ACT_SOFTMAX, 0, qo, gdpa.GDPA_ERR_INVALID_ARG),
                             (ACT_SOFTMAX, 8, np.array([0, 65], np.int32), gdpa.GDPA_ERR_INVALID_ARG)):
        with pytest.raises(gdpa.GdpaError) as e:
            gdpa.gdpa_fwd_sliding(0, 0, 0, qo, ko, 0, 0, 1, 1, 64, act, W, 1.0, 0)
        assert e.value.code == code


@pytest.mark.parametrize("W", [17, 256])
def test_sliding_window_planned_matches_the_async_entry(W):
    """gdpa_plan_create_sliding + gdpa_fwd_planned give the bits of
    gdpa_fwd_sliding (same items, same kernel), twice in a row with one plan."""
    rng = np.random.default_rng(8200 + W)
    L = np.array(LENGTHS)
    b = small_batch(rng, L, L, 2, 128, window_blocks=-W)
    w = b.workload
    ref = run_sliding(b, W, guard=0, as_tensor=True).clone()
    q, k, v = dev(b.q), dev(b.k), dev(b.v)
    qo = torch.from_numpy(b.q_offsets).cuda()
    ko = torch.from_numpy(b.kv_offsets).cuda()
    B = len(b.q_offsets) - 1
    plan = gdpa.gdpa_plan_create_sliding(b.q_offsets, b.kv_offsets, B, w.H, w.D, w.act, W)
    try:
        for _ in range(2):
            out = torch.full_like(ref, float("nan"))
            gdpa.gdpa_fwd_planned(plan, q, k, v, qo, ko, w.scale, out)
            assert gdpa.gdpa_device_status() == gdpa.GDPA_OK
            torch.cuda.synchronize()
            assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    finally:
        torch.cuda.synchronize()
        gdpa.gdpa_plan_destroy(plan)
    assert_parity(ref.float().cpu().numpy().astype(np.float64), oracle.gdpa_fwd_batch(b), "planned W=%d" % W)
