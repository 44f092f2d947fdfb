"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Bar (tests/parity.py): max |gpu - oracle| <= 1e-2 and relative L2 error
<= 5e-3, gpu output in bf16, oracle in fp64 on the same bf16 inputs; the
few-key edge cases add 2U|o| (U = 2^-8) to the absolute part, the two bf16
roundings of a one-key row.  Small cases and the five full-size workloads
(in the launch configuration the benchmark times) are compared element by
element over the whole output.
"""
from __future__ import annotations

import time

import numpy as np
import pytest
import torch

import oracle
from jagged_attention_recommender_gb300 import build as gbuild
from jagged_attention_recommender_gb300 import gdpa
from jagged_attention_recommender_gb300.workloads import (
    ACT_GELU_TANH, ACT_SILU, ACT_SOFTMAX, WORKLOADS, bf16_bits_to_f64, make_batch)
from tests.helpers import small_batch
from tests.parity import assert_parity, full_output_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    gbuild.build()
    yield


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.cuda()


def out_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def run_gpu(batch, entry="fwd", guard_rows=0):
    """Runs the CUDA path; returns fp64 [Tq, H, D] (and checks guard bands)."""
    w = batch.workload
    H, D = w.H, w.D
    Tq = int(batch.q_offsets[-1])
    q, k, v = dev_bf16(batch.q), dev_bf16(batch.k), dev_bf16(batch.v)
    qo = torch.from_numpy(batch.q_offsets).cuda()
    ko = torch.from_numpy(batch.kv_offsets).cuda()
    B = len(batch.q_offsets) - 1
    full = torch.full((Tq + 2 * guard_rows, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = full[guard_rows:guard_rows + Tq]
    if entry == "fwd":
        gdpa.gdpa_fwd(q, k, v, qo, ko, B, H, D, w.act, w.window_blocks, w.scale, out)
    elif entry == "async":
        gdpa.gdpa_fwd_async(q, k, v, batch.q_offsets, batch.kv_offsets, qo, ko, B, H, D, w.act, w.window_blocks,
                            w.scale, out)
    elif entry == "planned":
        plan = gdpa.gdpa_plan_create(batch.q_offsets, batch.kv_offsets, B, H, D, w.act, w.window_blocks)
        gdpa.gdpa_fwd_planned(plan, q, k, v, qo, ko, w.scale, out)
        torch.cuda.synchronize()
        gdpa.gdpa_plan_destroy(plan)
    elif entry == "host":
        hq = torch.from_numpy(batch.q.view(np.int16)).pin_memory()
        hk = torch.from_numpy(batch.k.view(np.int16)).pin_memory()
        hv = torch.from_numpy(batch.v.view(np.int16)).pin_memory()
        ho = torch.empty((Tq, H, D), dtype=torch.int16).pin_memory()
        gdpa.gdpa_fwd_host(hq, hk, hv, batch.q_offsets, batch.kv_offsets, B, H, D, w.act, w.window_blocks,
                           w.scale, ho)
        torch.cuda.synchronize()
        return bf16_bits_to_f64(ho.numpy().view(np.uint16))
    assert gdpa.gdpa_device_status() == gdpa.GDPA_OK
    torch.cuda.synchronize()
    if guard_rows:
        g = torch.cat([full[:guard_rows], full[guard_rows + Tq:]])
        assert torch.isnan(g.float()).all(), "kernel wrote outside its output rows"
    res = out_to_f64(out)
    return res


# ------------------------------------------------------------------ activation functions

ROUTES = {"sfu": gdpa.GDPA_ROUTE_SFU, "alu": gdpa.GDPA_ROUTE_ALU}


@pytest.fixture(params=list(ROUTES))
def route(request):
    """Runs the test under each sigma route of the GELU / SiLU activations."""
    gdpa.gdpa_set_act_route(ROUTES[request.param])
    yield request.param
    gdpa.gdpa_set_act_route(gdpa.GDPA_ROUTE_SFU)


def test_alu_gelu_within_1e3_of_exact_tanh_gelu(route):
    xs = torch.linspace(-17.0, 17.0, 1 << 20, dtype=torch.float32, device="cuda")
    ys = torch.empty_like(xs)
    gdpa.gdpa_act_eval(gdpa.GDPA_ACT_GELU_TANH, xs, ys)
    torch.cuda.synchronize()
    x64 = xs.cpu().double()
    ref = torch.nn.functional.gelu(x64, approximate="tanh")
    d = (ys.cpu().double() - ref).abs()
    assert d.max().item() <= 1e-3
    if route == "alu":
        assert d.max().item() <= 2e-6  # far inside the bar: the polynomial is accurate to fp32 level
    else:
        # ex2.approx and rcp.approx each keep about 22 bits; with the fp32
        # roundings of the cubic, 1 + e and the products the result is within
        # 2^-20 of |gelu(x)| <= |x| relative, and sigma's slope damps the
        # cubic's rounding further: allow 2^-19 |x| + 2^-24
        assert (d <= 2.0 ** -19 * x64.abs() + 2.0 ** -24).all()
    # outside the guaranteed range it saturates to x (x > 0) or 0 (x < 0)
    big = torch.tensor([20.0, 40.0, 1e3, -20.0, -40.0], device="cuda")
    yb = torch.empty_like(big)
    gdpa.gdpa_act_eval(gdpa.GDPA_ACT_GELU_TANH, big, yb)
    torch.cuda.synchronize()
    np.testing.assert_allclose(yb.cpu().numpy(), [20.0, 40.0, 1e3, 0.0, 0.0], atol=1e-4, rtol=1e-6)


def test_oracle_gelu_agrees_with_device_polynomial_on_grid(route):
    xs = np.linspace(-17.0, 17.0, 4001)
    ref = np.array([oracle.gelu_tanh(x) for x in xs])
    xt = torch.from_numpy(xs.astype(np.float32)).cuda()
    yt = torch.empty_like(xt)
    gdpa.gdpa_act_eval(gdpa.GDPA_ACT_GELU_TANH, xt, yt)
    torch.cuda.synchronize()
    # inputs are rounded to fp32 first: compare against the oracle at the rounded inputs
    ref32 = np.array([oracle.gelu_tanh(float(x)) for x in xs.astype(np.float32)])
    assert np.abs(yt.cpu().numpy() - ref32).max() <= 1e-3
    assert np.abs(ref32 - ref).max() < 1e-5


def test_alu_silu_matches_oracle_on_grid(route):
    # the kernels' SiLU: the GELU's sigma evaluation with A = 1, C = 0 (either route)
    x = np.linspace(-20.0, 20.0, 8001).astype(np.float32)
    xd = torch.from_numpy(x).cuda()
    y = torch.empty_like(xd)
    gdpa.gdpa_act_eval(ACT_SILU, xd, y)
    torch.cuda.synchronize()
    got = y.cpu().numpy().astype(np.float64)
    ref = np.array([oracle.silu(float(v)) for v in x])
    assert np.abs(got - ref).max() <= 1e-5 * np.maximum(1.0, np.abs(ref)).max()


# ------------------------------------------------------------------ small cases, element by element

SMALL = {
    # name: (B override) -- same distributions as the full workloads, several tiles and ragged tails
    "tiny": None,
    "pffn": 3,
    "self_long": 6,
    "cross_gelu": 5,
    "pma": 12,
    "block_window": 3,
}


@pytest.mark.parametrize("name", list(SMALL))
def test_small_workload_parity(name):
    batch = make_batch(name, B=SMALL[name], seed=WORKLOADS[name].seed + 100)
    ref = oracle.gdpa_fwd_batch(batch)
    got = run_gpu(batch, guard_rows=7)
    assert_parity(got, ref, name)


EDGE_LENGTHS = [0, 1, 63, 64, 65, 127, 128, 129, 200, 257]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("H", [1, 2, 8])
def test_edge_lengths_softmax_self(D, H):
    rng = np.random.default_rng(1000 + D + H)
    L = np.array(EDGE_LENGTHS)
    b = small_batch(rng, L, L, H, D)
    assert_parity(run_gpu(b, guard_rows=3), oracle.gdpa_fwd_batch(b), "edge D=%d H=%d" % (D, H))


@pytest.mark.parametrize("D", [64, 128])
def test_edge_lengths_cross_gelu(D):
    rng = np.random.default_rng(2000 + D)
    Lq = np.array([1, 129, 300, 0, 64, 77, 128])
    Lkv = np.array([0, 1, 8, 5, 64, 65, 300])  # empty KV, one key, several K/V tiles
    b = small_batch(rng, Lq, Lkv, 2, D, act=ACT_GELU_TANH, qk_norm=True, scale=1.0)
    assert_parity(run_gpu(b, guard_rows=3), oracle.gdpa_fwd_batch(b), "cross gelu D=%d" % D, few_keys=True)


@pytest.mark.parametrize("name", ["cross_gelu", "cross_silu", "pffn"])
def test_alu_route_parity(name):
    """The ALU-only sigma route (the polynomial of the GDPA section) through
    the forward kernels: same bar as the default route."""
    gdpa.gdpa_set_act_route(gdpa.GDPA_ROUTE_ALU)
    try:
        batch = make_batch(name, B=4, seed=WORKLOADS[name].seed + 300)
        got = run_gpu(batch, guard_rows=5)
    finally:
        gdpa.gdpa_set_act_route(gdpa.GDPA_ROUTE_SFU)
    assert_parity(got, oracle.gdpa_fwd_batch(batch), name + " (ALU route)")
    rng = np.random.default_rng(2100)
    Lq = np.array([1, 129, 300, 0, 64, 77, 128])
    Lkv = np.array([0, 1, 8, 5, 64, 65, 300])
    act = ACT_SILU if name == "cross_silu" else ACT_GELU_TANH
    b = small_batch(rng, Lq, Lkv, 2, 128, act=act, qk_norm=True, scale=1.0)
    gdpa.gdpa_set_act_route(gdpa.GDPA_ROUTE_ALU)
    try:
        got = run_gpu(b, guard_rows=3)
    finally:
        gdpa.gdpa_set_act_route(gdpa.GDPA_ROUTE_SFU)
    assert_parity(got, oracle.gdpa_fwd_batch(b), name + " edge lengths (ALU route)", few_keys=True)


@pytest.mark.parametrize("D", [64, 128])
def test_cross_softmax_long_kv(D):
    rng = np.random.default_rng(3000 + D)
    Lq = np.array([32, 32, 32, 5])
    Lkv = np.array([1000, 129, 4100, 0])
    b = small_batch(rng, Lq, Lkv, 3, D)
    assert_parity(run_gpu(b, guard_rows=3), oracle.gdpa_fwd_batch(b), "pma-like D=%d" % D)


@pytest.mark.parametrize("D", [64, 128])
def test_silu_cross_and_self(D):
    rng = np.random.default_rng(2500 + D)
    for Lq, Lkv in ((np.array([1, 129, 300, 0, 64, 77, 128]), np.array([0, 1, 8, 5, 64, 65, 300])),
                    (np.array([300, 257, 129, 500]), np.array([300, 257, 129, 500]))):
        b = small_batch(rng, Lq, Lkv, 2, D, act=ACT_SILU, qk_norm=True, scale=1.0)
        assert_parity(run_gpu(b, guard_rows=3), oracle.gdpa_fwd_batch(b), "silu D=%d" % D, few_keys=True)


def test_silu_key_split():
    rng = np.random.default_rng(2600)
    b = small_batch(rng, np.array(KS_LQ), np.array(KS_LKV), 2, 64, act=ACT_SILU, qk_norm=True, scale=1.0)
    assert_parity(run_gpu(b, guard_rows=3), oracle.gdpa_fwd_batch(b), "silu key split", few_keys=True)


# Short key ranges (every sequence at most 64 keys, one partial K/V tile):
# key counts around the 16-key MMA granule and the 32-column chunks, query
# counts around the 128-row tile and the 256-row item.
SK_LQ = [1, 127, 128, 129, 300, 1000, 40, 77, 5]
SK_LKV = [1, 15, 16, 17, 33, 63, 64, 0, 48]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("act", [ACT_SOFTMAX, ACT_GELU_TANH])
def test_short_kv_edges(D, act):
    rng = np.random.default_rng(3400 + D + act)
    gelu = act == ACT_GELU_TANH
    b = small_batch(rng, np.array(SK_LQ), np.array(SK_LKV), 3, D, act=act, qk_norm=gelu,
                    scale=1.0 if gelu else None)
    assert_parity(run_gpu(b, guard_rows=3), oracle.gdpa_fwd_batch(b), "short kv D=%d act=%d" % (D, act),
                  few_keys=gelu)


# Two-tile (256-row) items with 128-key K/V tiles (long key ranges) and with
# 64-key tiles (short key ranges): query counts around the 128/256-row edges,
# key counts around both tile sizes.
PAIR_LQ = [256, 257, 511, 300, 700, 129, 1000, 383]
PAIR_KV = {128: [256, 257, 511, 300, 700, 129, 1000, 383],
           64: [64, 65, 200, 1, 255, 129, 500, 0]}


@pytest.mark.parametrize("kv_tile", [128, 64])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("act", [ACT_SOFTMAX, ACT_GELU_TANH])
def test_pair_items(kv_tile, D, act):
    rng = np.random.default_rng(3600 + kv_tile + D + act)
    gelu = act == ACT_GELU_TANH
    b = small_batch(rng, np.array(PAIR_LQ), np.array(PAIR_KV[kv_tile]), 2, D, act=act, qk_norm=gelu,
                    scale=1.0 if gelu else None)
    _, _, _, rows, kvt = gdpa.gdpa_plan_enumerate(b.q_offsets, b.kv_offsets, b.B, 2, D, act, 0, 8, with_rows=True)
    assert (rows, kvt) == (256, kv_tile)
    assert_parity(run_gpu(b, guard_rows=3), oracle.gdpa_fwd_batch(b), "pair kv_tile=%d D=%d act=%d"
                  % (kv_tile, D, act), few_keys=gelu)


# Key-split items (D = 64, every sequence at most 32 queries): the four
# activation warps share the queries and split each K/V tile into 32-key
# blocks; key counts around the block and tile edges, and query counts below
# and at 32.
KS_LQ = [1, 7, 31, 32, 32, 5, 32, 32, 17, 32, 32, 32, 2, 32]
KS_LKV = [1, 31, 32, 33, 95, 96, 97, 127, 128, 129, 255, 256, 0, 1000]


@pytest.mark.parametrize("H", [1, 3, 8])
def test_key_split_edges_softmax(H):
    rng = np.random.default_rng(3100 + H)
    b = small_batch(rng, np.array(KS_LQ), np.array(KS_LKV), H, 64)
    items, _, _, rows, _ = gdpa.gdpa_plan_enumerate(b.q_offsets, b.kv_offsets, b.B, H, 64, 0, 0, 8, with_rows=True)
    assert rows == 32
    assert_parity(run_gpu(b, guard_rows=3), oracle.gdpa_fwd_batch(b), "key split H=%d" % H)


def test_key_split_edges_gelu():
    rng = np.random.default_rng(3200)
    b = small_batch(rng, np.array(KS_LQ), np.array(KS_LKV), 2, 64, act=ACT_GELU_TANH, qk_norm=True, scale=1.0)
    assert_parity(run_gpu(b, guard_rows=3), oracle.gdpa_fwd_batch(b), "key split gelu", few_keys=True)


def test_key_split_merges_blocks_with_far_apart_maxima():
    # Each 32-key block of a tile has its own running max; blocks whose keys
    # score 0, 20 and 60 (scale 1) must merge by 2^(m_k - M) exactly, and
    # later tiles raise the max again (lazy rescale inside one warp).
    from tests.helpers import bits, with_values
    rng = np.random.default_rng(3300)
    Lkv, H, D = 520, 2, 64
    b = small_batch(rng, [32, 9], [Lkv, Lkv], H, D, scale=1.0)
    q = np.ones((41, H, D), np.float32)
    k = rng.standard_normal((2 * Lkv, H, D)).astype(np.float32) * 0.01
    for s0 in (0, Lkv):
        k[s0 + 32:s0 + 64] += 20.0 / D
        k[s0 + 100:s0 + 128] += 60.0 / D
        k[s0 + 300:s0 + 310] += 90.0 / D
    b = with_values(b, q=bits(q), k=bits(k))
    assert_parity(run_gpu(b), oracle.gdpa_fwd_batch(b), "key split maxima")


@pytest.mark.parametrize("wb", [1, 2, 4, 7])
def test_window_variants(wb):
    rng = np.random.default_rng(4000 + wb)
    L = np.array([1, 64, 65, 200, 640, 1000])  # includes partial tail blocks
    b = small_batch(rng, L, L, 2, 128, window_blocks=wb)
    assert_parity(run_gpu(b, guard_rows=3), oracle.gdpa_fwd_batch(b), "window %d" % wb)


def test_window_d64():
    rng = np.random.default_rng(4100)
    L = np.array([128, 384, 333])
    b = small_batch(rng, L, L, 4, 64, window_blocks=4)
    assert_parity(run_gpu(b), oracle.gdpa_fwd_batch(b), "window D=64")


@pytest.mark.parametrize("jump", [16.0, 64.0, 96.0])
def test_softmax_score_jumps_between_key_tiles(jump):
    # Keys of the first 128-key tile score 0, later keys score `jump` (scale 1):
    # the running max rises by jump*log2(e) between tiles.  16 takes the
    # deferred rescale, 64 and 96 overrun the single pass and redo the tile.
    # Enough queries per sequence to take the two-tile items.
    from tests.helpers import bits
    rng = np.random.default_rng(5100)
    L, H, D = 300, 1, 64
    b = small_batch(rng, [L, L], [L, L], H, D, scale=1.0)
    q = np.ones((2 * L, H, D), np.float32)
    k = np.zeros((2 * L, H, D), np.float32)
    for s0 in (0, L):
        k[s0 + 128:s0 + L] = jump / D
    from tests.helpers import with_values
    b = with_values(b, q=bits(q), k=bits(k))
    got = run_gpu(b)
    ref = oracle.gdpa_fwd_batch(b)
    assert_parity(got, ref, "jump %g" % jump)


def test_zero_and_negative_scale():
    rng = np.random.default_rng(5000)
    for scale in (0.0, -0.09):
        b = small_batch(rng, [70, 130], [70, 130], 2, 64, scale=scale)
        assert_parity(run_gpu(b), oracle.gdpa_fwd_batch(b), "scale %g" % scale)


def test_all_entry_points_agree_and_are_deterministic():
    batch = make_batch("self_long", B=4, seed=77)
    a = run_gpu(batch, "fwd")
    b = run_gpu(batch, "planned")
    c = run_gpu(batch, "host")
    d = run_gpu(batch, "fwd")
    e = run_gpu(batch, "async")
    assert np.array_equal(a, b) and np.array_equal(a, c) and np.array_equal(a, d) and np.array_equal(a, e)


def test_host_entry_pipelines_chunks_exactly():
    # ~300 MB in + out: the host entry point splits it into several chunks of
    # whole sequences; every item computes exactly as in the one-shot launch.
    batch = make_batch("self_long", B=64, seed=78)
    a = run_gpu(batch, "fwd")
    c = run_gpu(batch, "host")
    assert np.array_equal(a, c)
    sub = batch.subset(sample_sequences(batch, 3, 5))
    assert_parity(run_gpu(sub, "host"), oracle.gdpa_fwd_batch(sub), "host chunks")


def test_empty_batch_is_noop():
    rng = np.random.default_rng(6000)
    b = small_batch(rng, [0, 0], [3, 0], 2, 64)
    got = run_gpu(b)
    assert got.shape == (0, 2, 64)


# ------------------------------------------------------------------ full-size workloads, every row

def sample_sequences(batch, n, seed):
    Lq, _ = batch.lengths()
    rng = np.random.default_rng(seed)
    B = len(Lq)
    pick = {int(np.argmax(Lq)), int(np.argmin(Lq))}
    while len(pick) < min(n, B):
        pick.add(int(rng.integers(0, B)))
    return sorted(pick)


def run_gpu_async(batch):
    """The benchmark's call (gdpa_fwd_async, host plan + upload + kernel); returns the device output."""
    w = batch.workload
    Tq = int(batch.q_offsets[-1])
    q, k, v = dev_bf16(batch.q), dev_bf16(batch.k), dev_bf16(batch.v)
    qo = torch.from_numpy(batch.q_offsets).cuda()
    ko = torch.from_numpy(batch.kv_offsets).cuda()
    out = torch.full((Tq, w.H, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    gdpa.gdpa_fwd_async(q, k, v, batch.q_offsets, batch.kv_offsets, qo, ko, batch.B, w.H, w.D, w.act,
                        w.window_blocks, w.scale, out)
    assert gdpa.gdpa_device_status() == gdpa.GDPA_OK
    torch.cuda.synchronize()
    del q, k, v
    return out


@pytest.mark.parametrize("name", ["tiny", "self_long", "cross_gelu", "pma", "block_window"])
def test_full_workload_parity(name):
    """Every row of the full-size workload, in the benchmark's launch, against the oracle."""
    batch = make_batch(name)
    out = run_gpu_async(batch)
    worst, rl2, rows = full_output_parity(batch, lambda t0, t1: out_to_f64(out[t0:t1]), oracle.gdpa_fwd_batch,
                                          name)
    assert rows == int(batch.q_offsets[-1])
    print("%s: %d rows, max |d| %.2e, rel L2 %.2e" % (name, rows, worst, rl2))


# ------------------------------------------------------------------ failure path

def test_bounded_wait_times_out_and_context_survives():
    assert gdpa.gdpa_device_status() == gdpa.GDPA_OK
    t0 = time.perf_counter()
    gdpa.gdpa_wait_selftest(200)
    st = gdpa.gdpa_device_status()
    dt = time.perf_counter() - t0
    assert st == gdpa.GDPA_ERR_DEVICE_TIMEOUT
    assert 0.15 < dt < 5.0
    assert gdpa.gdpa_device_status() == gdpa.GDPA_OK  # the word was cleared
    # the context is still usable: a normal forward pass still matches the oracle
    batch = make_batch("tiny", seed=91)
    assert_parity(run_gpu(batch), oracle.gdpa_fwd_batch(batch), "after timeout")
