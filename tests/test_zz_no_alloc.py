"""gdpa_fwd_noalloc, the entry point for callers that must not allocate.

Serving processes that carve device memory into a fixed arena, or framework
hooks that must stay inside their own caching allocator, cannot let the
library call cudaMalloc.  gdpa_fwd_noalloc keeps its work list in a fixed
device array instead.  These tests call it through the C ABI on every kernel
path the planner can pick -- 256-row items on 128-key tiles (self_long) and
on 64-key tiles (cross_gelu), key-split items (a pma-shaped D = 64 batch),
block windows, and single-tile items (tiny) -- two calls in a row each,
larger batches first, so a stale tail of the shared array from an earlier
call must not leak into a later one.  Each output is compared with gdpa_fwd's
and with the fp64 oracle at the parity bar (tests/parity.py).  The file is
named to be collected last.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from jagged_attention_recommender_gb300 import build as gbuild
from jagged_attention_recommender_gb300 import gdpa
from jagged_attention_recommender_gb300.workloads import make_batch
from tests.parity import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    gbuild.build()
    yield


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _run(entry, batch):
    w = batch.workload
    q, k, v = _dev(batch.q), _dev(batch.k), _dev(batch.v)
    qo = torch.from_numpy(batch.q_offsets).cuda()
    ko = torch.from_numpy(batch.kv_offsets).cuda()
    out = torch.full((int(batch.q_offsets[-1]), w.H, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    entry(q, k, v, qo, ko, batch.B, w.H, w.D, w.act, w.window_blocks, w.scale, out)
    assert gdpa.gdpa_device_status() == gdpa.GDPA_OK
    return out.float().cpu().numpy().astype(np.float64)


def _check(batch, what):
    got = _run(gdpa.gdpa_fwd_noalloc, batch)
    assert_parity(got, _run(gdpa.gdpa_fwd, batch), what + " vs gdpa_fwd")
    assert_parity(got, oracle.gdpa_fwd_batch(batch), what + " vs oracle")


def test_noalloc_matches_gdpa_fwd_on_two_calls_in_a_row():
    big = make_batch("self_long", B=12, seed=501)    # more work items first ...
    small = make_batch("cross_gelu", B=2, seed=502)  # ... then fewer, another kernel path
    for batch in (big, small):
        _check(batch, batch.workload.name)


def test_noalloc_key_split_and_block_window_paths():
    # pma-shaped (D = 64, 32 queries per sequence: key-split items), then a
    # block window (256-row window items on 64-key tiles), then single-tile items
    for batch in (make_batch("pma", B=24, seed=503), make_batch("block_window", B=2, seed=504),
                  make_batch("tiny", seed=505)):
        _, _, _, rows, _ = gdpa.gdpa_plan_enumerate(batch.q_offsets, batch.kv_offsets, batch.B, batch.workload.H,
                                                    batch.workload.D, batch.workload.act,
                                                    batch.workload.window_blocks, 8, with_rows=True)
        assert rows == {"pma": 32, "block_window": 256, "tiny": 128}[batch.workload.name]
        _check(batch, batch.workload.name)


def test_noalloc_rejects_batches_beyond_its_limit():
    with pytest.raises(gdpa.GdpaError) as e:  # B above the 65536-sequence limit, before any GPU work
        gdpa.gdpa_fwd_noalloc(0, 0, 0, 0, 0, 70000, 1, 64, 0, 0, 1.0, 0)
    assert e.value.code == gdpa.GDPA_ERR_NO_MEMORY
