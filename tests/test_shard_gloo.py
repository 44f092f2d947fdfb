"""Multi-rank path on CPU: world_size-2 gloo processes each take their LPT
shard of one jagged batch (whole sequences, rebased offsets), compute it
with the oracle, and the reassembled output equals the unsharded run
exactly.  No data moves between ranks except this test's own gather."""
from __future__ import annotations

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from jagged_attention_recommender_gb300.shard import partition_sequences, scatter_rows, shard
from jagged_attention_recommender_gb300.workloads import make_batch


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, name, B, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle

        batch = make_batch(name, B=B, seed=31)
        fwd = oracle.gdpa_fwd_mx_batch if batch.workload.mx else oracle.gdpa_fwd_batch
        sub, seqs = shard(batch, rank, world)
        out = fwd(sub, nthreads=2)
        gathered = [None] * world if rank == 0 else None
        dist.gather_object((seqs, out), gathered, dst=0)
        if rank == 0:
            full = fwd(batch, nthreads=2)
            got = np.full_like(full, np.nan)
            all_seqs = []
            for s, o in gathered:
                scatter_rows(full.shape[0], batch, s, o, got)
                all_seqs += s
            ok = sorted(all_seqs) == list(range(batch.B)) and np.array_equal(got, full)
            q.put(("ok" if ok else "mismatch", len(gathered[0][0]), len(gathered[1][0])))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("name,B", [("self_long", 6), ("block_window", 3), ("cross_gelu", 5), ("self_long_mx", 6)])
def test_two_rank_shards_reassemble_exactly(name, B):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, name, B, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    assert all(p.exitcode == 0 for p in procs)
    res = q.get(timeout=5)
    assert res[0] == "ok", res
    assert res[1] > 0 and res[2] > 0


def test_partition_is_balanced_and_complete():
    rng = np.random.default_rng(3)
    L = np.clip(np.round(rng.lognormal(6.9, 0.8, 256)), 100, 4096).astype(np.int64)
    parts = partition_sequences(L, L, 8)
    flat = sorted(s for p in parts for s in p)
    assert flat == list(range(256))
    loads = [sum(int(L[s]) ** 2 for s in p) for p in parts]
    assert max(loads) / (sum(loads) / 8) < 1.05


def test_bench_shards_one_seeded_batch_per_rank():
    # bench.py under torchrun: rank r times its LPT shard of one global batch
    # of N x B sequences; the shards' lengths together are the global draw
    import bench
    from jagged_attention_recommender_gb300.workloads import WORKLOADS, draw_lengths

    w = WORKLOADS["tiny"]
    world = 3
    Lq, Lkv = draw_lengths(w, np.random.default_rng(w.seed), w.B * world)
    got_q, flops = [], None
    for r in range(world):
        b, per_rank = bench.bench_batch("tiny", r, world)
        got_q += list(np.diff(b.q_offsets))
        flops = per_rank if flops is None else flops
        assert per_rank == flops
        assert abs(bench.useful_flops(b) - per_rank[r]) < 1e-6
    assert sorted(got_q) == sorted(Lq.tolist())
    single, per1 = bench.bench_batch("tiny", 0, 1)
    assert per1 == [bench.useful_flops(single)] and single.B == w.B
