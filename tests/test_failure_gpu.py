"""Failure paths on the GPU, made on the host or by a bounded wait -- no
fault, trap or hang.

* An allocation that fails (the library's buffer growth, forced through the
  test-only environment variable GDPA_FAULT_INJECT=alloc) makes the call
  return GDPA_ERR_NO_MEMORY before any GPU work; the next call succeeds.
* A plan used with device offsets it was not built from, reaching past the
  tensors: the kernel clips every item to the rows that exist, writes
  nothing outside `out` (NaN guard rows stay NaN) and flags the launch, so
  gdpa_device_status returns GDPA_ERR_INVALID_ARG; the next call is exact.
* A real forward launch whose bounded wait runs out: with
  GDPA_FAULT_INJECT=skip_arrive one activation warp of CTA 0 withholds its
  arrival on the first item's O-free barrier, the MMA warp's wait gives up
  after GDPA_WAIT_TIMEOUT_MS, every role stops and drains (copies waited
  for, MMAs committed, tensor memory freed), and the launch reports
  GDPA_ERR_DEVICE_TIMEOUT; a following forward in the same context matches
  the oracle.  Run in a child process so that its short wait limit does not
  apply to the other tests.
"""
from __future__ import annotations

import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from jagged_attention_recommender_gb300 import build as gbuild
from jagged_attention_recommender_gb300 import gdpa
from jagged_attention_recommender_gb300.workloads import make_batch, offsets_of
from tests.parity import assert_parity

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    gbuild.build()
    yield


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def test_allocation_failure_is_reported_and_the_next_call_succeeds():
    batch = make_batch("self_long", B=3, seed=701)
    w = batch.workload
    q, k, v = _dev(batch.q), _dev(batch.k), _dev(batch.v)
    qo = torch.from_numpy(batch.q_offsets).cuda()
    ko = torch.from_numpy(batch.kv_offsets).cuda()
    out = torch.full((int(batch.q_offsets[-1]), w.H, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    os.environ["GDPA_FAULT_INJECT"] = "alloc"
    try:
        with pytest.raises(gdpa.GdpaError) as e:
            gdpa.gdpa_fwd(q, k, v, qo, ko, batch.B, w.H, w.D, w.act, 0, w.scale, out)
        assert e.value.code == gdpa.GDPA_ERR_NO_MEMORY
        with pytest.raises(gdpa.GdpaError) as e:
            gdpa.gdpa_fwd_async(q, k, v, batch.q_offsets, batch.kv_offsets, qo, ko, batch.B, w.H, w.D, w.act, 0,
                                w.scale, out)
        assert e.value.code == gdpa.GDPA_ERR_NO_MEMORY
    finally:
        del os.environ["GDPA_FAULT_INJECT"]
    assert gdpa.gdpa_device_status() == gdpa.GDPA_OK
    assert torch.isnan(out.float()).all()  # the failed calls launched nothing
    gdpa.gdpa_fwd(q, k, v, qo, ko, batch.B, w.H, w.D, w.act, 0, w.scale, out)
    assert gdpa.gdpa_device_status() == gdpa.GDPA_OK
    assert_parity(_f64(out), oracle.gdpa_fwd_batch(batch), "after the failed allocation")


@pytest.mark.parametrize("name", ["self_long", "cross_gelu", "tiny"])
def test_plan_with_offsets_past_the_tensors_is_flagged_and_stays_inside(name):
    # one plan per kernel family: 256-row items on 128-key tiles, on 64-key
    # tiles, and single-tile items
    batch = make_batch(name, B=4, seed=702)
    w = batch.workload
    Tq, Tkv = int(batch.q_offsets[-1]), int(batch.kv_offsets[-1])
    guard = 5
    q, k, v = _dev(batch.q), _dev(batch.k), _dev(batch.v)
    full = torch.full((Tq + 2 * guard, w.H, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = full[guard:guard + Tq]
    plan = gdpa.gdpa_plan_create(batch.q_offsets, batch.kv_offsets, batch.B, w.H, w.D, w.act, 0)
    try:
        # device offsets whose sequences run past both tensors
        Lq, Lkv = batch.lengths()
        bad_q = torch.from_numpy(offsets_of(Lq * 2 + 7)).cuda()
        bad_k = torch.from_numpy(offsets_of(Lkv * 2 + 7)).cuda()
        gdpa.gdpa_fwd_planned(plan, q, k, v, bad_q, bad_k, w.scale, out)
        assert gdpa.gdpa_device_status() == gdpa.GDPA_ERR_INVALID_ARG
        g = torch.cat([full[:guard], full[guard + Tq:]])
        assert torch.isnan(g.float()).all(), "a bad plan wrote outside out"
        assert gdpa.gdpa_device_status() == gdpa.GDPA_OK  # the flag was cleared
        # the same plan with the offsets it was built from is exact
        qo = torch.from_numpy(batch.q_offsets).cuda()
        ko = torch.from_numpy(batch.kv_offsets).cuda()
        gdpa.gdpa_fwd_planned(plan, q, k, v, qo, ko, w.scale, out)
        assert gdpa.gdpa_device_status() == gdpa.GDPA_OK
    finally:
        torch.cuda.synchronize()
        gdpa.gdpa_plan_destroy(plan)
    assert Tkv > 0
    assert_parity(_f64(out), oracle.gdpa_fwd_batch(batch), name + " after the bad plan", few_keys=w.act != 0)


_CHILD = r"""
import json, os, sys, time
import numpy as np, torch
sys.path.insert(0, %(root)r)
import oracle
from jagged_attention_recommender_gb300 import gdpa
from jagged_attention_recommender_gb300.workloads import make_batch
batch = make_batch("self_long", B=96, seed=703)
w = batch.workload
dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
q, k, v = dev(batch.q), dev(batch.k), dev(batch.v)
qo = torch.from_numpy(batch.q_offsets).cuda(); ko = torch.from_numpy(batch.kv_offsets).cuda()
out = torch.empty((int(batch.q_offsets[-1]), w.H, w.D), dtype=torch.bfloat16, device="cuda")
_, _, _, rows, kvt = gdpa.gdpa_plan_enumerate(batch.q_offsets, batch.kv_offsets, batch.B, w.H, w.D, w.act, 0,
                                               torch.cuda.get_device_properties(0).multi_processor_count, with_rows=True)
os.environ["GDPA_FAULT_INJECT"] = "skip_arrive"
t0 = time.perf_counter()
gdpa.gdpa_fwd_async(q, k, v, batch.q_offsets, batch.kv_offsets, qo, ko, batch.B, w.H, w.D, w.act, 0, w.scale, out)
st1 = gdpa.gdpa_device_status()
dt = time.perf_counter() - t0
del os.environ["GDPA_FAULT_INJECT"]
gdpa.gdpa_fwd_async(q, k, v, batch.q_offsets, batch.kv_offsets, qo, ko, batch.B, w.H, w.D, w.act, 0, w.scale, out)
st2 = gdpa.gdpa_device_status()
got = out.float().cpu().numpy().astype(np.float64)
ref = oracle.gdpa_fwd_batch(batch)
d = float(np.abs(got - ref).max())
rl2 = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
print(json.dumps({"st1": st1, "st2": st2, "dt": dt, "max_abs": d, "rel_l2": rl2, "rows": rows, "kv_tile": kvt}))
"""


def test_forward_wait_runs_out_drains_and_the_next_forward_is_exact():
    env = dict(os.environ, GDPA_WAIT_TIMEOUT_MS="300")
    env.pop("GDPA_FAULT_INJECT", None)
    r = subprocess.run([sys.executable, "-c", _CHILD % {"root": ROOT}], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert (res["rows"], res["kv_tile"]) == (256, 128)  # the 128-key pair kernel, where the hook sits
    assert res["st1"] == gdpa.GDPA_ERR_DEVICE_TIMEOUT
    assert 0.25 < res["dt"] < 30.0
    assert res["st2"] == gdpa.GDPA_OK
    assert res["max_abs"] <= 1e-2 and res["rel_l2"] <= 5e-3, res
