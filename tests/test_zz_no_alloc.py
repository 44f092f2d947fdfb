"""gdpa_fwd_noalloc, the entry point for callers that must not allocate.

Serving processes that carve device memory into a fixed arena, or framework
hooks that must stay inside their own caching allocator, cannot let the
library call cudaMalloc.  gdpa_fwd_noalloc keeps its work list in a fixed
device array instead.  These tests call it through the C ABI twice in a row
-- a larger batch, then a smaller one, so a stale tail of the shared array
from the first call must not leak into the second -- and compare each output
with gdpa_fwd's within the parity tolerance (max |d| <= 1e-2, rel-L2 <= 5e-3).
The file is named to be collected last.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from jagged_attention_recommender_gb300 import build as gbuild
from jagged_attention_recommender_gb300 import gdpa
from jagged_attention_recommender_gb300.workloads import make_batch

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


def _close(a, b):
    assert np.isfinite(a).all()
    assert np.abs(a - b).max() <= 1e-2
    assert np.linalg.norm(a - b) <= 5e-3 * max(np.linalg.norm(b), 1e-30)


def test_noalloc_matches_gdpa_fwd_on_two_calls_in_a_row():
    big = make_batch("self_long", B=12, seed=501)    # more work items first ...
    small = make_batch("cross_gelu", B=2, seed=502)  # ... then fewer, another kernel path
    for batch in (big, small):
        _close(_run(gdpa.gdpa_fwd_noalloc, batch), _run(gdpa.gdpa_fwd, batch))


def test_noalloc_rejects_batches_beyond_its_limit():
    with pytest.raises(gdpa.GdpaError) as e:  # B above the 65536-sequence limit, before any GPU work
        gdpa.gdpa_fwd_noalloc(0, 0, 0, 0, 0, 70000, 1, 64, 0, 0, 1.0, 0)
    assert e.value.code == gdpa.GDPA_ERR_NO_MEMORY
