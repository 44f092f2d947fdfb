"""GPU parity of the training path: gdpa_fwd_lse's row logsumexp and
gdpa_bwd's dq, dk, dv against the fp64 oracle (tests/test_oracle_bwd_pins.py
pins the oracle).

The bar, from the arithmetic: P and dS enter the tensor cores as bf16
(relative rounding up to 2^-9), O enters <dO, O> as the forward's bf16
output (2^-9), and every product of a gradient sum carries at most ~2^-8
relative error before the fp32 accumulation; dS = P (dP - <dO, O>) cancels,
so the error scales with the tensor's magnitude rather than each element's.
Per tensor: max |d| <= 2^-6 max |ref| and rel-L2 <= 1e-2.  The row
logsumexp is fp32 arithmetic on the fp32 scores: |d| <= 2e-3.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from jagged_attention_recommender_gb300 import build as gbuild, gdpa
from jagged_attention_recommender_gb300.workloads import (
    ACT_GELU_TANH, ACT_SILU, ACT_SOFTMAX, WORKLOADS, bf16_bits_to_f64, make_batch)
from tests.helpers import bits, small_batch

pytestmark = pytest.mark.gpu

MAX_REL = 2.0 ** -6
REL_L2 = 1e-2
LSE_ABS = 2e-3


@pytest.fixture(scope="module", autouse=True)
def built():
    gbuild.build()
    yield


def dev(bits_arr):
    return torch.from_numpy(np.ascontiguousarray(bits_arr).view(np.int16)).view(torch.bfloat16).cuda()


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def rand_dout(rng, batch):
    w = batch.workload
    return bits(rng.standard_normal((int(batch.q_offsets[-1]), w.H, w.D)).astype(np.float32))


def run_train(batch, dout, guard=0):
    """Forward with lse, then backward, on the GPU.  Returns fp64 out, lse, dq, dk, dv."""
    w = batch.workload
    H, D, B = w.H, w.D, len(batch.q_offsets) - 1
    Tq, Tkv = int(batch.q_offsets[-1]), int(batch.kv_offsets[-1])
    q, k, v, do = dev(batch.q), dev(batch.k), dev(batch.v), dev(dout)
    qo = torch.from_numpy(batch.q_offsets).cuda()
    ko = torch.from_numpy(batch.kv_offsets).cuda()
    out = torch.full((Tq, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((Tq, H), float("nan"), dtype=torch.float32, device="cuda")
    if w.window_blocks < 0:  # sliding window of -window_blocks tokens
        gdpa.gdpa_fwd_sliding(q, k, v, batch.q_offsets, batch.kv_offsets, qo, ko, B, H, D, w.act, -w.window_blocks,
                              w.scale, out, lse)
    else:
        gdpa.gdpa_fwd_lse(q, k, v, batch.q_offsets, batch.kv_offsets, qo, ko, B, H, D, w.act, w.window_blocks,
                          w.scale, out, lse)
    nan = float("nan")
    dq_full = torch.full((Tq + 2 * guard, H, D), nan, dtype=torch.bfloat16, device="cuda")
    dk_full = torch.full((Tkv + 2 * guard, H, D), nan, dtype=torch.bfloat16, device="cuda")
    dv_full = torch.full((Tkv + 2 * guard, H, D), nan, dtype=torch.bfloat16, device="cuda")
    dq, dk, dv = dq_full[guard:guard + Tq], dk_full[guard:guard + Tkv], dv_full[guard:guard + Tkv]
    if w.window_blocks < 0:
        gdpa.gdpa_bwd_sliding(q, k, v, out, do, lse, batch.q_offsets, batch.kv_offsets, qo, ko, B, H, D, w.act,
                              -w.window_blocks, w.scale, dq, dk, dv)
    else:
        gdpa.gdpa_bwd(q, k, v, out, do, lse, batch.q_offsets, batch.kv_offsets, qo, ko, B, H, D, w.act,
                      w.window_blocks, w.scale, dq, dk, dv)
    assert gdpa.gdpa_device_status() == gdpa.GDPA_OK
    torch.cuda.synchronize()
    if guard:
        for full, T in ((dq_full, Tq), (dk_full, Tkv), (dv_full, Tkv)):
            g = torch.cat([full[:guard], full[guard + T:]])
            assert torch.isnan(g.float()).all(), "backward wrote outside its rows"
    return f64(out), lse.cpu().numpy().astype(np.float64), f64(dq), f64(dk), f64(dv)


def assert_grad(got, ref, what):
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), "non-finite " + what
    if not ref.size:
        return
    scale = float(np.abs(ref).max())
    d = np.abs(got - ref)
    if scale == 0.0:
        # exact zeros by cancellation (e.g. a one-key window: dS = P (dP - <dO, O>)
        # with o = v); the GPU forms dP in the tensor core and <dO, O> in the
        # prep kernel, whose fp32 sums of D products differ by ~2^-24 D |dO||v|
        assert d.max() <= 1e-4, "%s: expected zeros, max |d| %.3e" % (what, d.max())
        return
    assert d.max() <= MAX_REL * scale, "%s: max |d| %.3e vs bar %.3e" % (what, d.max(), MAX_REL * scale)
    rl2 = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert rl2 <= REL_L2, "%s: rel L2 %.3e" % (what, rl2)


def check(batch, seed, guard=3):
    rng = np.random.default_rng(seed)
    do = rand_dout(rng, batch)
    out, lse, dq, dk, dv = run_train(batch, do, guard)
    rq, rk, rv, rl = oracle.gdpa_bwd_batch(batch, do)
    if batch.workload.act == ACT_SOFTMAX:
        fin = np.isfinite(rl)
        assert np.array_equal(np.isfinite(lse), fin), "lse: empty-row pattern"
        assert np.abs(lse[fin] - rl[fin]).max(initial=0.0) <= LSE_ABS
    assert_grad(dq, rq, "dq")
    assert_grad(dk, rk, "dk")
    assert_grad(dv, rv, "dv")


# Ragged self attention: lengths around the 128-row / 128-key tile edges.
EDGE = [1, 63, 127, 128, 129, 200, 257, 300]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("H", [1, 3])
def test_bwd_softmax_self_ragged(D, H):
    rng = np.random.default_rng(6000 + D + H)
    L = np.array(EDGE)
    check(small_batch(rng, L, L, H, D), 6100 + D + H)


@pytest.mark.parametrize("D", [64, 128])
def test_bwd_softmax_cross_and_empty(D):
    # cross attention, a sequence without keys (dq = 0) and one without
    # queries (dk = dv = 0)
    rng = np.random.default_rng(6200 + D)
    Lq = np.array([40, 0, 300, 129, 7, 256])
    Lkv = np.array([500, 77, 0, 16, 1, 130])
    check(small_batch(rng, Lq, Lkv, 2, D), 6300 + D)


@pytest.mark.parametrize("route", ["sfu", "alu"])
@pytest.mark.parametrize("D", [64, 128])
def test_bwd_gelu(D, route):
    # both sigma routes (gdpa_set_act_route) through the forward and the backward
    rng = np.random.default_rng(6400 + D)
    Lq = np.array([129, 33, 300, 0, 64])
    Lkv = np.array([40, 200, 8, 9, 128])
    gdpa.gdpa_set_act_route(gdpa.GDPA_ROUTE_ALU if route == "alu" else gdpa.GDPA_ROUTE_SFU)
    try:
        check(small_batch(rng, Lq, Lkv, 2, D, act=ACT_GELU_TANH, qk_norm=True, scale=1.0), 6500 + D)
    finally:
        gdpa.gdpa_set_act_route(gdpa.GDPA_ROUTE_SFU)


@pytest.mark.parametrize("D", [64, 128])
def test_bwd_silu(D):
    rng = np.random.default_rng(6450 + D)
    Lq = np.array([129, 33, 300, 0, 64])
    Lkv = np.array([40, 200, 8, 9, 128])
    check(small_batch(rng, Lq, Lkv, 2, D, act=ACT_SILU, qk_norm=True, scale=1.0), 6550 + D)


def test_bwd_zero_scale_and_negative_scale():
    rng = np.random.default_rng(6600)
    for scale in (0.0, -0.09):
        check(small_batch(rng, [70, 130], [70, 130], 2, 64, scale=scale), 6700)


@pytest.mark.parametrize("name", ["self_long", "cross_gelu"])
def test_bwd_small_workloads(name):
    batch = make_batch(name, B=4, seed=WORKLOADS[name].seed + 200)
    check(batch, 6800)


def test_fwd_lse_keeps_the_forward_output():
    batch = make_batch("self_long", B=5, seed=77)
    w = batch.workload
    H, D, B = w.H, w.D, len(batch.q_offsets) - 1
    Tq = int(batch.q_offsets[-1])
    q, k, v = dev(batch.q), dev(batch.k), dev(batch.v)
    qo = torch.from_numpy(batch.q_offsets).cuda()
    ko = torch.from_numpy(batch.kv_offsets).cuda()
    a = torch.empty((Tq, H, D), dtype=torch.bfloat16, device="cuda")
    b = torch.empty_like(a)
    lse = torch.empty((Tq, H), dtype=torch.float32, device="cuda")
    gdpa.gdpa_fwd(q, k, v, qo, ko, B, H, D, w.act, w.window_blocks, w.scale, a)
    gdpa.gdpa_fwd_lse(q, k, v, batch.q_offsets, batch.kv_offsets, qo, ko, B, H, D, w.act, w.window_blocks, w.scale,
                      b, lse)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_fwd_lse_all_kernels():
    # the key-split single-tile kernel (D = 64, <= 32 queries), the 64-key pair
    # kernel (short keys) and the block window each write the logsumexp
    rng = np.random.default_rng(6900)
    cases = [small_batch(rng, [32, 5, 0, 17], [1000, 40, 3, 0], 3, 64),
             small_batch(rng, [300, 400], [40, 100], 2, 128),
             small_batch(rng, [130, 640, 65], [130, 640, 65], 2, 128, window_blocks=3)]
    for batch in cases:
        w = batch.workload
        H, D, B = w.H, w.D, len(batch.q_offsets) - 1
        Tq = int(batch.q_offsets[-1])
        q, k, v = dev(batch.q), dev(batch.k), dev(batch.v)
        qo = torch.from_numpy(batch.q_offsets).cuda()
        ko = torch.from_numpy(batch.kv_offsets).cuda()
        out = torch.empty((Tq, H, D), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((Tq, H), float("nan"), dtype=torch.float32, device="cuda")
        gdpa.gdpa_fwd_lse(q, k, v, batch.q_offsets, batch.kv_offsets, qo, ko, B, H, D, w.act, w.window_blocks,
                          w.scale, out, lse)
        torch.cuda.synchronize()
        got = lse.cpu().numpy().astype(np.float64)
        ref = oracle.gdpa_bwd_batch(batch, np.zeros_like(batch.q))[3]
        fin = np.isfinite(ref)
        assert np.array_equal(np.isfinite(got), fin)
        assert np.abs(got[fin] - ref[fin]).max(initial=0.0) <= LSE_ABS


def test_bwd_full_self_long_every_row():
    # the full workload in the launch the bench times, every row of dq, dk,
    # dv and the lse against the oracle, group by group of whole sequences
    # (sequences are independent, so their gradients are too); the per-tensor
    # bar uses the whole tensor's max |ref|, as the small cases do
    from tests.parity import sequence_groups
    batch = make_batch("self_long")
    rng = np.random.default_rng(7000)
    do = rand_dout(rng, batch)
    out, lse, dq, dk, dv = run_train(batch, do)
    qo, ko = batch.q_offsets, batch.kv_offsets
    stats = {n: [0.0, 0.0, 0.0, 0.0] for n in ("dq", "dk", "dv")}  # max|d|, max|ref|, sum d^2, sum ref^2
    rows = 0
    for seqs in sequence_groups(qo, 1 << 15):
        sub = batch.subset(seqs)
        sq = slice(int(qo[seqs[0]]), int(qo[seqs[-1] + 1]))
        sk = slice(int(ko[seqs[0]]), int(ko[seqs[-1] + 1]))
        rq, rk, rv, rl = oracle.gdpa_bwd_batch(sub, do[sq])
        assert np.abs(lse[sq] - rl).max(initial=0.0) <= LSE_ABS
        for n, got, ref in (("dq", dq[sq], rq), ("dk", dk[sk], rk), ("dv", dv[sk], rv)):
            assert np.isfinite(got).all(), "non-finite " + n
            st = stats[n]
            d = np.abs(got - ref)
            st[0] = max(st[0], float(d.max(initial=0.0)))
            st[1] = max(st[1], float(np.abs(ref).max(initial=0.0)))
            st[2] += float(np.sum(d * d))
            st[3] += float(np.sum(ref * ref))
        rows += sq.stop - sq.start
    assert rows == int(qo[-1])
    for n, (dmax, rmax, dd, rr) in stats.items():
        assert dmax <= MAX_REL * rmax, "%s: max |d| %.3e vs bar %.3e" % (n, dmax, MAX_REL * rmax)
        assert np.sqrt(dd / rr) <= REL_L2, "%s: rel L2 %.3e" % (n, np.sqrt(dd / rr))


# Windows: lengths around the 64-token blocks and the 128-row / 64-row tiles.
WIN_L = [1, 64, 65, 200, 640, 1000, 130]


@pytest.mark.parametrize("W", [1, 2, 4])
@pytest.mark.parametrize("D", [64, 128])
def test_bwd_block_window(W, D):
    rng = np.random.default_rng(7100 + 10 * W + D)
    L = np.array(WIN_L)
    check(small_batch(rng, L, L, 2, D, window_blocks=W), 7200 + W + D)


@pytest.mark.parametrize("W", [1, 64, 100, 300])
def test_bwd_sliding_window(W):
    rng = np.random.default_rng(7300 + W)
    L = np.array(WIN_L)
    check(small_batch(rng, L, L, 2, 128, window_blocks=-W), 7400 + W)


def test_bwd_rejects_bad_windows():
    qo = np.array([0, 64], np.int32)
    with pytest.raises(gdpa.GdpaError) as e:  # windows are softmax only
        gdpa.gdpa_bwd(0, 0, 0, 0, 0, 0, qo, qo, 0, 0, 1, 1, 64, ACT_GELU_TANH, 2, 1.0, 0, 0, 0)
    assert e.value.code == gdpa.GDPA_ERR_UNSUPPORTED
    with pytest.raises(gdpa.GdpaError) as e:
        gdpa.gdpa_bwd_sliding(0, 0, 0, 0, 0, 0, qo, qo, 0, 0, 1, 1, 64, ACT_SOFTMAX, 0, 1.0, 0, 0, 0)
    assert e.value.code == gdpa.GDPA_ERR_INVALID_ARG
