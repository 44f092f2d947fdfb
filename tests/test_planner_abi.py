"""Host-side tests of libgdpa (no GPU): the C ABI loads and exports every
declared symbol, argument validation, and the jagged tile planner
(coverage, key ranges, load balance)."""
from __future__ import annotations

import os
import re

import numpy as np
import pytest

from jagged_attention_recommender_gb300 import build as gbuild
from jagged_attention_recommender_gb300 import gdpa
from jagged_attention_recommender_gb300.workloads import WORKLOADS, draw_lengths, offsets_of

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    gbuild.build()
    yield


def header_functions():
    src = open(os.path.join(ROOT, "include", "gdpa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gdpa_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    names = header_functions()
    assert set(names) == set(gdpa.EXPORTS)
    L = gdpa.lib()
    for n in names:
        assert hasattr(L, n), n
    assert gdpa.gdpa_version().startswith("gdpa")
    assert gdpa.gdpa_status_string(0) == "GDPA_OK"
    assert gdpa.gdpa_status_string(4) == "GDPA_ERR_DEVICE_TIMEOUT"
    assert gdpa.gdpa_status_string(99) == "GDPA_ERR_UNKNOWN"


def test_sliding_plan_argument_checks_need_no_gpu():
    qo = np.array([0, 64], np.int32)
    for act, W, ko, code in ((0, 0, qo, gdpa.GDPA_ERR_INVALID_ARG),
                             (0, -5, qo, gdpa.GDPA_ERR_INVALID_ARG),
                             (1, 8, qo, gdpa.GDPA_ERR_UNSUPPORTED)):
        with pytest.raises(gdpa.GdpaError) as e:
            gdpa.gdpa_plan_create_sliding(qo, ko, 1, 1, 64, act, W)
        assert e.value.code == code


def test_act_route_setter_needs_no_gpu():
    assert gdpa.gdpa_get_act_route() == gdpa.GDPA_ROUTE_SFU  # the default
    try:
        gdpa.gdpa_set_act_route(gdpa.GDPA_ROUTE_ALU)
        assert gdpa.gdpa_get_act_route() == gdpa.GDPA_ROUTE_ALU
        for bad in (-1, 2, 7):
            with pytest.raises(gdpa.GdpaError) as e:
                gdpa.gdpa_set_act_route(bad)
            assert e.value.code == gdpa.GDPA_ERR_INVALID_ARG
            assert gdpa.gdpa_get_act_route() == gdpa.GDPA_ROUTE_ALU  # unchanged
    finally:
        gdpa.gdpa_set_act_route(gdpa.GDPA_ROUTE_SFU)
    assert gdpa.gdpa_get_act_route() == gdpa.GDPA_ROUTE_SFU


def test_shape_validation_needs_no_gpu():
    # rejected before any CUDA call
    with pytest.raises(gdpa.GdpaError) as e:
        gdpa.gdpa_fwd(0, 0, 0, 0, 0, 1, 1, 96, 0, 0, 1.0, 0, stream=0)
    assert e.value.code == gdpa.GDPA_ERR_UNSUPPORTED
    with pytest.raises(gdpa.GdpaError) as e:
        gdpa.gdpa_fwd(0, 0, 0, 0, 0, 1, 0, 64, 0, 0, 1.0, 0, stream=0)
    assert e.value.code == gdpa.GDPA_ERR_INVALID_ARG
    with pytest.raises(gdpa.GdpaError) as e:  # GELU with a window is not implemented
        gdpa.gdpa_fwd(0, 0, 0, 0, 0, 1, 1, 64, 1, 2, 1.0, 0, stream=0)
    assert e.value.code == gdpa.GDPA_ERR_UNSUPPORTED
    with pytest.raises(gdpa.GdpaError) as e:
        gdpa.gdpa_fwd(0, 0, 0, 0, 0, 1, 1, 64, 7, 0, 1.0, 0, stream=0)
    assert e.value.code == gdpa.GDPA_ERR_INVALID_ARG
    # an empty batch is a no-op
    gdpa.gdpa_fwd(0, 0, 0, 0, 0, 0, 1, 64, 0, 0, 1.0, 0, stream=0)


def test_mx_argument_checks_need_no_gpu():
    # gdpa_fwd_mx: D other than 128, a misaligned or missing scale pointer, a
    # bad activation -- all rejected before any CUDA call
    qo = np.array([0, 64], np.int32)
    for D, q_sf, act, code in ((64, 256, 0, gdpa.GDPA_ERR_UNSUPPORTED), (128, 257, 0, gdpa.GDPA_ERR_INVALID_ARG),
                               (128, 0, 0, gdpa.GDPA_ERR_INVALID_ARG), (128, 256, 9, gdpa.GDPA_ERR_INVALID_ARG)):
        with pytest.raises(gdpa.GdpaError) as e:
            gdpa.gdpa_fwd_mx(256, q_sf, 256, 256, 256, qo, qo, 0, 0, 1, 1, D, act, 1.0, 256, stream=0)
        assert e.value.code == code
    gdpa.gdpa_fwd_mx(0, 0, 0, 0, 0, np.zeros(1, np.int32), np.zeros(1, np.int32), 0, 0, 0, 1, 128, 0, 1.0, 0, stream=0)


def test_enumerate_rejects_bad_offsets():
    for qo, ko, wb in [([0, 5, 3], [0, 1, 2], 0),   # decreasing
                       ([1, 5], [0, 5], 0),         # not starting at 0
                       ([0, 5], [0, 4], 2)]:        # window needs equal offsets
        with pytest.raises(gdpa.GdpaError) as e:
            gdpa.gdpa_plan_enumerate(qo, ko, len(qo) - 1, 2, 64, 0, wb, 8)
        assert e.value.code == gdpa.GDPA_ERR_INVALID_ARG


def check_plan(Lq, Lkv, H, wb, num_ctas):
    qo, ko = offsets_of(Lq), offsets_of(Lkv)
    B = len(Lq)
    items, cta, cost, R, kvt = gdpa.gdpa_plan_enumerate(qo, ko, B, H, 128, 0, wb, num_ctas, with_rows=True)
    n = len(items)
    busy = Lq > 0
    if wb > 0:
        expect_R = 256 if busy.any() else 128  # the two tiles' windows overlap
    else:
        expect_R = 256 if (busy.any() and Lq[busy].sum() > 128 * busy.sum()) else 128
    assert R == expect_R
    # 256-row items stage 64-key tiles for windows and short key ranges
    # (at most 256 keys per busy sequence on average), 128-key tiles otherwise
    if R != 256:
        expect_kvt = 128
    elif wb > 0 or Lkv[busy].sum() <= 256 * busy.sum():
        expect_kvt = 64
    else:
        expect_kvt = 128
    assert kvt == expect_kvt
    # CSR over CTAs
    assert cta[0] == 0 and cta[-1] == n and np.all(np.diff(cta) >= 0)
    # every (sequence, head, query row) is covered exactly once
    cover = {}
    for (b, h, q0, kv0) in items:
        assert 0 <= b < B and 0 <= h < H and q0 % R == 0 and 0 <= q0 < Lq[b]
        key = (int(b), int(h), int(q0))
        assert key not in cover
        cover[key] = int(kv0)
    expect = {(b, h, q0) for b in range(B) for h in range(H) for q0 in range(0, int(Lq[b]), R)}
    assert set(cover) == expect
    # key ranges: full attention starts at 0; a window tile starts at the first
    # key any of its rows may see
    for (b, h, q0), kv0 in cover.items():
        if wb == 0:
            assert kv0 == 0
        else:
            assert kv0 == max(0, (q0 // 64 - (wb - 1)) * 64)
    # greedy list scheduling bound: max load <= mean load + largest item
    loads = np.array([cost[cta[c]:cta[c + 1]].sum() for c in range(num_ctas)])
    if n:
        assert loads.max() <= cost.sum() / num_ctas + cost.max()
        # LPT order inside each CTA: non-increasing cost
        for c in range(num_ctas):
            seg = cost[cta[c]:cta[c + 1]]
            assert np.all(np.diff(seg) <= 0)
    return items, cta, cost, loads


@pytest.mark.parametrize("seed", range(4))
def test_plan_coverage_random(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 40))
    Lq = rng.integers(0, 700, size=B)
    Lkv = rng.integers(0, 700, size=B)
    check_plan(Lq, Lkv, int(rng.integers(1, 5)), 0, int(rng.integers(1, 20)))


@pytest.mark.parametrize("wb", [1, 2, 4, 9])
def test_plan_coverage_window(wb):
    rng = np.random.default_rng(wb)
    L = rng.integers(0, 900, size=13)
    check_plan(L, L, 2, wb, 7)


def test_plan_empty_sequences():
    items, cta, cost, _ = check_plan(np.array([0, 0, 5]), np.array([3, 0, 0]), 2, 0, 4)  # average 5 rows: R = 128
    assert len(items) == 2 and set(items[:, 0]) == {2}


def test_short_query_batches_take_key_split_items():
    # D = 64, full attention, every sequence at most 32 queries: one 32-row
    # item per (sequence, head); otherwise the window / 128 / 256-row rules
    qo, ko = offsets_of(np.array([32, 0, 5, 32])), offsets_of(np.array([900, 40, 0, 3000]))
    items, cta, cost, R, _ = gdpa.gdpa_plan_enumerate(qo, ko, 4, 3, 64, 0, 0, 5, with_rows=True)
    assert R == 32
    assert sorted(map(tuple, items[:, :3].tolist())) == sorted((b, h, 0) for b in (0, 2, 3) for h in range(3))
    assert np.all(items[:, 3] == 0) and cta[-1] == len(items)
    # cost grows with the key range
    by_seq = {int(b): c for (b, _, _, _), c in zip(items, cost)}
    assert by_seq[3] > by_seq[0] > by_seq[2]
    for D, wb, lq, R_want in ((128, 0, 32, 128), (64, 2, 32, 256), (64, 0, 33, 128), (64, 0, 300, 256)):
        q2 = offsets_of(np.array([lq, lq]))
        _, _, _, R2, _ = gdpa.gdpa_plan_enumerate(q2, q2, 2, 1, D, 0, wb, 4, with_rows=True)
        assert R2 == R_want


def test_plan_balances_the_long_jagged_workload():
    w = WORKLOADS["self_long"]
    Lq, Lkv = draw_lengths(w, np.random.default_rng(w.seed))
    _, _, cost, loads = check_plan(Lq, Lkv, w.H, 0, 152)
    # skew (max / mean CTA load) stays close to 1
    assert loads.max() / loads.mean() < 1.05


def lpt_reference(Lq, Lkv, H, R, num_ctas, cost_of):
    """The planner's schedule restated in plain Python: items in (sequence,
    query tile, head) order, a stable sort by decreasing cost // 16, each item
    to the least-loaded CTA (the lowest index among equals), items of a CTA in
    that order."""
    items = [(b, h, q0) for b in range(len(Lq)) for q0 in range(0, int(Lq[b]), R) for h in range(H)]
    cost = [cost_of[(b, q0)] for (b, h, q0) in items]
    order = sorted(range(len(items)), key=lambda i: -(cost[i] >> 4))  # sorted() is stable
    load = [0] * num_ctas
    per = [[] for _ in range(num_ctas)]
    for i in order:
        c = min(range(num_ctas), key=lambda k: (load[k], k))
        load[c] += cost[i]
        per[c].append(i)
    flat = [items[i] for c in range(num_ctas) for i in per[c]]
    cta = np.cumsum([0] + [len(p) for p in per])
    return flat, cta


@pytest.mark.parametrize("huge,ctas", [(False, 7), (True, 7), (False, 150), (False, 131)])
def test_plan_matches_plain_lpt_schedule(huge, ctas):
    # huge key counts make the cost buckets outnumber the items, which takes
    # the in-place sort instead of the counting sort: both must give the
    # schedule of the plain restatement, exactly.  With 7 CTAs the items
    # outnumber twice the tree's leaves (the packed-key tree); with 131 or 150
    # CTAs they do not (the general tree): both give the same schedule.
    rng = np.random.default_rng(99 + huge + ctas)
    B, H = 23, 3
    Lq = rng.integers(0, 600, size=B)
    Lkv = rng.integers(0, 600, size=B) * (5000 if huge else 1)
    qo, ko = offsets_of(Lq), offsets_of(Lkv)
    items, cta, cost, R, _ = gdpa.gdpa_plan_enumerate(qo, ko, B, H, 128, 0, 0, ctas, with_rows=True)
    if huge:
        assert int(cost.max()) >> 4 > 4 * len(items) + 1026
    cost_of = {(int(b), int(q0)): int(c) for (b, _, q0, _), c in zip(items, cost)}
    flat, cta_ref = lpt_reference(Lq, Lkv, H, R, ctas, cost_of)
    assert np.array_equal(cta, cta_ref)
    assert [tuple(map(int, (b, h, q0))) for (b, h, q0, _) in items] == flat
