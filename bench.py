#!/usr/bin/env python3
"""Throughput benchmark of the jagged GDPA forward pass on GB300.

One step = the whole forward path over one batch of the workload: host tile
planning from the batch's offsets, work-list upload, and the persistent
tcgen05 kernel (``gdpa_fwd_async`` through the C ABI).  Inputs are resident
in HBM before the timed region; the workload's inputs (Q, K, V ~1 GB for the
default workload) are larger than the 126 MB L2, so no L2 flush is done
between steps.

Prints one JSON line (rank 0).  ``value`` is useful TFLOPS: 4*D*H per
unmasked (query, key) pair, summed over all ranks, over the max-over-ranks
time.  With the default workload (self_long, the headline) the line also
carries a ``workloads`` object: the other configurations of the metric
(tiny, cross_gelu, pma, block_window), each timed the same way with its own
roofline, end-to-end figure and clock record.  Under torchrun each rank
takes its LPT shard (whole sequences) of one seeded global batch of N times
the workload's sequences, so per-GPU work stays about fixed (weak scaling)
and no data moves between ranks.  ``--impl reference`` times the fp64 CPU
oracle instead (the slow baseline arm) on a bounded sample of the same
workload.

``--pass backward`` times the training backward instead (``gdpa_bwd``: dq,
dk, dv from the forward's output and row logsumexp, which are computed once
before the timed region); its useful FLOPs are the five products of the
backward, 10*D*H per unmasked pair (2.5 times the forward's).
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from jagged_attention_recommender_gb300.metrics import algorithmic_bytes, useful_flops  # noqa: E402
from jagged_attention_recommender_gb300.workloads import ACT_SOFTMAX, WORKLOADS, make_batch  # noqa: E402

METRIC = "jagged GDPA fwd useful TFLOPS (unpadded) & % of GB300 roofline, 1 GPU"
METRIC_BWD = "jagged GDPA bwd useful TFLOPS (unpadded, 10*D*H per pair) & % of GB300 roofline, 1 GPU"
DEFAULT_WORKLOAD = "self_long"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

RECIPES = {
    "tiny": "B=4 H=2 D=64, L~U{1..128}, softmax, scale=1/sqrt(D)",
    "self_long": "B=256 H=4 D=128, L=clip(round(lognormal(6.9,0.8)),100,4096), softmax non-causal, scale=1/sqrt(D)",
    "cross_gelu": "B=512 H=4 D=128, Lq~U{256..4096}, Lkv~U{8..64}, QK-normed x4, GELU-tanh, scale=1, /Lkv",
    "pma": "B=256 H=8 D=64, 32 shared seed queries per sample, Lkv=clip(round(lognormal(7.6,1.0)),100,16384), softmax",
    "block_window": "B=64 H=4 D=128, L=64*U{8..512}, 64-token blocks, window 4 blocks (own causal + 3 previous), softmax",
    "sliding_window": "B=64 H=4 D=128, L~U{512..32768}, causal sliding window of 256 tokens, softmax",
    "cross_silu": "B=512 H=4 D=128, Lq~U{256..4096}, Lkv~U{8..64}, QK-normed x4, SiLU, scale=1, /Lkv",
    "pffn": "B=256 H=4 D=128, Lq~U{256..4096}, 512 hidden units per sample as keys/values, GELU-tanh, scale=1/sqrt(D)",
    "self_long_mx": "self_long with Q, K, V in MXFP8 (e4m3, E8M0 scale per 32 of D for Q/K, per 32 keys for V, "
                    "V key-major) and P rounded to MXFP8 on chip; both products on the block-scaled e4m3 MMA; O bf16",
}
BOUND = {"tiny": "hbm", "self_long": "tensor", "cross_gelu": "hbm", "pma": "hbm", "block_window": "hbm",
         "sliding_window": "hbm", "cross_silu": "hbm", "pffn": "tensor", "self_long_mx": "tensor"}
# All-MXFP8 forward: Q K^T and P V both on the e4m3 tensor core, nominally
# twice the bf16 rate (4.5 vs 2.25 PFLOP/s dense)
MX_PEAK_FACTOR = 2.0


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="target CPU time of the oracle baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="time the headline workload only (skip the other configurations of the metric)")
    ap.add_argument("--pass", dest="pass_", choices=["forward", "backward"], default="forward")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# Source files each forward kernel is compiled from (the shared headers plus
# its own); the hash keys the committed ncu traffic figure to the kernel.
KERNEL_SOURCES = {
    "gdpa_fwd_pair_kernel": ["gdpa_fwd_common.cuh", "sm103_ptx.cuh", "gelu_alu.cuh", "gdpa_fwd_pair.cuh"],
    "gdpa_fwd_pair64_kernel": ["gdpa_fwd_common.cuh", "sm103_ptx.cuh", "gelu_alu.cuh", "gdpa_fwd_pair64.cuh"],
    "gdpa_fwd_kernel": ["gdpa_fwd_common.cuh", "sm103_ptx.cuh", "gelu_alu.cuh", "gdpa_fwd_kernel.cuh"],
    "gdpa_fwd_mxp_kernel": ["gdpa_fwd_common.cuh", "sm103_ptx.cuh", "gelu_alu.cuh", "gdpa_fwd_pair64.cuh",
                            "gdpa_fwd_mxp.cuh"],
}


def kernel_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "jagged_attention_recommender_gb300", "csrc", f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def kernel_for(batch, gdpa_mod, num_ctas: int) -> str:
    """The kernel the planner picks for this batch: 256-row items take a pair
    kernel (64- or 128-key K/V tiles), the rest the single-tile kernel."""
    w = batch.workload
    if w.window_blocks < 0:  # sliding windows: 256-row items on the 64-key pair kernel
        return "gdpa_fwd_pair64_kernel"
    if w.mx:  # all-MXFP8: 256-row items, 64-key score tiles
        return "gdpa_fwd_mxp_kernel"
    _, _, _, rows, kv_tile = gdpa_mod.gdpa_plan_enumerate(batch.q_offsets, batch.kv_offsets, batch.B, w.H, w.D,
                                                          w.act, w.window_blocks, num_ctas, with_rows=True)
    if rows != 256:
        return "gdpa_fwd_kernel"
    return "gdpa_fwd_pair64_kernel" if kv_tile == 64 else "gdpa_fwd_pair_kernel"


def traffic_per_launch(workload: str, kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this kernel's current source."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
        e = t.get(workload)
        if e and e.get("kernel") == kernel and e.get("kernel_hash") == kernel_hash(kernel):
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons), "samples": len(sm)}


def oracle_fwd(batch):
    import oracle

    return oracle.gdpa_fwd_mxfp8_batch(batch) if batch.workload.mx else oracle.gdpa_fwd_batch(batch)


def oracle_sample(batch, target_s: float, seed: int = 2024):
    """A seeded subset of whole sequences sized for ~target_s of oracle CPU time."""
    import oracle

    rng = np.random.default_rng(seed)
    order = rng.permutation(batch.B)
    # calibrate the oracle's rate on a first small slice
    probe = [int(order[0])]
    sub = batch.subset(probe)
    t0 = time.perf_counter()
    oracle_fwd(sub)
    dt = max(time.perf_counter() - t0, 1e-3)
    rate = useful_flops(sub) / dt  # single-sequence rate: at most H threads busy
    cores = oracle.num_cpus()
    rate_all = rate * max(1.0, min(cores, 4 * batch.H) / batch.H)
    want = rate_all * target_s
    seqs, acc = [], 0.0
    for s in order:
        f = useful_flops(batch.subset([int(s)]))
        seqs.append(int(s))
        acc += f
        if acc >= want:
            break
    return batch.subset(seqs), seqs


def time_oracle(sample, reps=1):
    import oracle

    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        oracle_fwd(sample)
        times.append(time.perf_counter() - t0)
    return times


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    import oracle

    w = WORKLOADS[args.workload]
    batch = make_batch(args.workload)
    total_steps = args.steps + args.warmup
    per_step = max(0.5, min(10.0, 150.0 / max(1, total_steps)))
    sample, seqs = oracle_sample(batch, per_step)
    flops = useful_flops(sample)
    for _ in range(args.warmup):
        time_oracle(sample)
    times = time_oracle(sample, args.steps)
    t = sum(times)
    value = flops * args.steps / t / 1e12
    cores = oracle.num_cpus()
    desc = "%d of %d sequences (seeded), all %d heads, %.3g useful GFLOP per step" % (
        len(seqs), batch.B, w.H, flops / 1e9)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "%s: %s" % (args.workload, RECIPES[args.workload]), "seed": w.seed,
                   "sample": desc},
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# The configurations of the target metric besides the headline one; each is
# timed the same way and reported under "workloads" in the JSON line.
METRIC_CONFIGS = ["tiny", "cross_gelu", "pma", "block_window"]
# and two more rows of the path: the headline workload with every input in
# MXFP8, and the token-granular sliding window
EXTRA_WORKLOADS = ["self_long_mx", "sliding_window", "pffn"]


def bench_batch(name: str, rank: int, world: int):
    """The rank's batch: at N = 1 the workload's seeded batch; at N > 1 the
    rank's LPT shard (whole sequences, shard.partition_sequences) of one
    seeded global batch of N times the workload's sequences, so per-GPU work
    stays about fixed (weak scaling) and no data moves between ranks.  Values
    are drawn for the rank's own sequences only.  Returns (batch, per-rank
    useful FLOPs of every rank)."""
    from jagged_attention_recommender_gb300.metrics import key_count
    from jagged_attention_recommender_gb300.shard import partition_sequences
    from jagged_attention_recommender_gb300.workloads import draw_lengths

    w = WORKLOADS[name]
    if world == 1:
        batch = make_batch(name)
        return batch, [useful_flops(batch)]
    Lq, Lkv = draw_lengths(w, np.random.default_rng(w.seed), w.B * world)
    parts = partition_sequences(Lq, Lkv, world, w.window_blocks)
    per_rank = [4.0 * w.D * w.H * sum(key_count(int(Lq[s]), int(Lkv[s]), w.window_blocks) for s in p)
                for p in parts]
    mine = parts[rank]
    return make_batch(name, seed=w.seed + 1000 * rank, lengths=(Lq[mine], Lkv[mine])), per_rank


def measure_forward(name, args, rank, world, local, dist, gdpa, with_e2e=True):
    """Times K steps of one workload's forward pass; returns the measurement dict."""
    import torch

    w = WORKLOADS[name]
    batch, per_rank = bench_batch(name, rank, world)
    flops = useful_flops(batch)
    nbytes = algorithmic_bytes(batch)
    H, D, B = w.H, w.D, batch.B
    Tq = int(batch.q_offsets[-1])

    def dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()

    q, k, v = dev(batch.q), dev(batch.k), dev(batch.v)
    qo = torch.from_numpy(batch.q_offsets).cuda()
    ko = torch.from_numpy(batch.kv_offsets).cuda()
    out = torch.empty((Tq, H, D), dtype=torch.bfloat16, device="cuda")
    h_qo, h_ko = batch.q_offsets, batch.kv_offsets
    stream = torch.cuda.current_stream()

    if w.mx:
        q8, qsf, k8, ksf, vt8, vtsf = (torch.from_numpy(np.ascontiguousarray(a)).cuda()
                                       for a in (batch.q8, batch.q_sf, batch.k8, batch.k_sf, batch.vt8, batch.vt_sf))

    def step():
        if w.window_blocks < 0:
            gdpa.gdpa_fwd_sliding(q, k, v, h_qo, h_ko, qo, ko, B, H, D, w.act, -w.window_blocks, w.scale, out, None,
                                  stream)
        elif w.mx:
            gdpa.gdpa_fwd_mxfp8(q8, qsf, k8, ksf, vt8, vtsf, h_qo, h_ko, qo, ko, B, H, D, w.act, w.scale, out, None,
                                stream)
        else:
            gdpa.gdpa_fwd_async(q, k, v, h_qo, h_ko, qo, ko, B, H, D, w.act, w.window_blocks, w.scale, out, stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    st = gdpa.gdpa_device_status()
    if st != gdpa.GDPA_OK:
        raise SystemExit("%s: device status after warm-up: %s" % (name, gdpa.gdpa_status_string(st)))

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                           else int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local]))
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    e0.record(stream)
    for i in range(K):
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    st = gdpa.gdpa_device_status()
    if st != gdpa.GDPA_OK:
        raise SystemExit("%s: device status after timing: %s" % (name, gdpa.gdpa_status_string(st)))
    elapsed_ms = e0.elapsed_time(e1)
    launch_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    if dist:
        t = torch.tensor([elapsed_ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed_ms = float(t.item())
    total_flops = float(sum(per_rank))
    value = total_flops * K / (elapsed_ms / 1e3) / 1e12

    # ---- end to end through the public C ABI with host buffers (H2D + compute + D2H each step):
    # gdpa_fwd_host where it applies (bf16, block windows), else the copies around the entry point
    e2e = None
    if with_e2e and w.window_blocks >= 0 and not w.mx:
        hq = torch.from_numpy(batch.q.view(np.int16)).pin_memory()
        hk = torch.from_numpy(batch.k.view(np.int16)).pin_memory()
        hv = torch.from_numpy(batch.v.view(np.int16)).pin_memory()
        ho = torch.empty((Tq, H, D), dtype=torch.int16).pin_memory()
        h2d = int(hq.numel() + hk.numel() + hv.numel()) * 2 + 2 * 4 * (B + 1)
        d2h = int(ho.numel()) * 2
        gdpa.gdpa_fwd_host(hq, hk, hv, h_qo, h_ko, B, H, D, w.act, w.window_blocks, w.scale, ho, stream)
        e2e_t = []
        for _ in range(max(1, args.e2e_steps)):
            if dist:
                dist.barrier()
            t0 = time.perf_counter()
            gdpa.gdpa_fwd_host(hq, hk, hv, h_qo, h_ko, B, H, D, w.act, w.window_blocks, w.scale, ho, stream)
            e2e_t.append(time.perf_counter() - t0)
        e2e_s = statistics.mean(e2e_t)
        if dist:
            t = torch.tensor([e2e_s], device="cuda")
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            e2e_s = float(t.item())
        e2e_value = total_flops / e2e_s / 1e12
        e2e = {"value": e2e_value, "unit": "TFLOPS", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_s * 1e3, "entry": "gdpa_fwd_host"}
        del hq, hk, hv, ho
    elif with_e2e:
        # the sliding-window and MXFP8 entry points take device tensors: each
        # step copies the inputs from pinned host memory, calls the entry
        # point and reads the output back, all on the stream
        if w.mx:
            host_in = [torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
                       for a in (batch.q8, batch.q_sf, batch.k8, batch.k_sf, batch.vt8, batch.vt_sf)]
            dev_in = [q8, qsf, k8, ksf, vt8, vtsf]
            entry = "H2D copies + gdpa_fwd_mxfp8 + D2H"
        else:
            host_in = [torch.from_numpy(a.view(np.int16)).pin_memory() for a in (batch.q, batch.k, batch.v)]
            dev_in = [q.view(torch.int16), k.view(torch.int16), v.view(torch.int16)]
            entry = "H2D copies + gdpa_fwd_sliding + D2H"
        h_qo_t = torch.from_numpy(batch.q_offsets).pin_memory()
        h_ko_t = torch.from_numpy(batch.kv_offsets).pin_memory()
        ho = torch.empty((Tq, H, D), dtype=torch.int16).pin_memory()
        h2d = int(sum(t.numel() * t.element_size() for t in host_in)) + 2 * 4 * (B + 1)
        d2h = int(ho.numel()) * 2

        def e2e_step():
            for hsrc, ddst in zip(host_in, dev_in):
                ddst.copy_(hsrc, non_blocking=True)
            qo.copy_(h_qo_t, non_blocking=True)
            ko.copy_(h_ko_t, non_blocking=True)
            step()
            ho.copy_(out.view(torch.int16), non_blocking=True)
            stream.synchronize()

        e2e_step()
        e2e_t = []
        for _ in range(max(1, args.e2e_steps)):
            if dist:
                dist.barrier()
            t0 = time.perf_counter()
            e2e_step()
            e2e_t.append(time.perf_counter() - t0)
        e2e_s = statistics.mean(e2e_t)
        if dist:
            t = torch.tensor([e2e_s], device="cuda")
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            e2e_s = float(t.item())
        e2e = {"value": total_flops / e2e_s / 1e12, "unit": "TFLOPS", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3, "entry": entry}
        del host_in, ho

    peaks, peak_src = load_peaks()
    bound = BOUND[name]
    if bound == "tensor":
        achieved = flops / (launch_ms / 1e3) / 1e12
        peak = peaks["bf16_tflops"] * (MX_PEAK_FACTOR if w.mx else 1.0)
        unit = "TFLOP/s"
    else:
        achieved = nbytes / (launch_ms / 1e3) / 1e9
        peak = peaks["hbm_gbs"]
        unit = "GB/s"
    kernel = kernel_for(batch, gdpa, torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count)
    traffic = traffic_per_launch(name, kernel) if world == 1 else None
    peak_note = " (burst)" if bound == "tensor" else ""
    if w.mx:
        peak_note = " (burst bf16 x 2: both products at the nominal e4m3 rate, twice bf16's)"
    roofline = {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
                "traffic": traffic, "peak_source": peak_src + peak_note,
                "launch_ms": launch_ms, "useful_flops_per_launch": flops, "algorithmic_bytes_per_launch": nbytes,
                "kernel": kernel, "kernel_hash": kernel_hash(kernel)}
    res = {"name": name, "batch": batch, "B": B, "Tq": Tq, "Tkv": int(batch.kv_offsets[-1]), "K": K,
           "elapsed_ms": elapsed_ms, "ms_per_step": elapsed_ms / K, "value": value, "clocks": clocks, "e2e": e2e,
           "roofline": roofline, "flops": flops, "per_rank_flops": per_rank,
           "input_gb": (q.numel() + k.numel() + v.numel()) * 2 / 1e9}
    del q, k, v, out, qo, ko
    torch.cuda.empty_cache()
    return res


def run_ours(args, rank, world, local):
    import torch

    from jagged_attention_recommender_gb300 import build as gbuild
    from jagged_attention_recommender_gb300 import gdpa

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    gbuild.build()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    head = measure_forward(args.workload, args, rank, world, local, dist, gdpa)
    w = WORKLOADS[args.workload]
    batch, B, Tq, K = head["batch"], head["B"], head["Tq"], head["K"]

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle

        sample, seqs = oracle_sample(batch, args.cpu_seconds)
        t = time_oracle(sample)[0]
        cpu = {"value": useful_flops(sample) / t / 1e12, "unit": "TFLOPS", "cores": oracle.num_cpus(),
               "kind": "oracle", "sample": "%d of %d sequences (seeded), all %d heads, %.3g useful GFLOP, %.1f s" % (
                   len(seqs), B, w.H, useful_flops(sample) / 1e9, t)}
    del head["batch"], batch

    others = {}
    if args.workload == DEFAULT_WORKLOAD and not args.no_workloads:
        for name in METRIC_CONFIGS + EXTRA_WORKLOADS:
            r = measure_forward(name, args, rank, world, local, dist, gdpa)
            others[name] = {"workload": "%s: %s" % (name, RECIPES[name]), "ms_per_step": r["ms_per_step"],
                            "dtype": "mxfp8 (Q, K, V, P) + bf16 O" if WORKLOADS[name].mx else "bf16",
                            "value": r["value"], "unit": "TFLOPS", "roofline": r["roofline"], "e2e": r["e2e"],
                            "clocks": r["clocks"], "tokens_q": r["Tq"], "tokens_kv": r["Tkv"],
                            "gpu_launches": r["K"]}
            del r
            if WORKLOADS[name].act != ACT_SOFTMAX:
                # the same launch with the ALU-only sigma route (the GDPA
                # section's polynomial) for comparison; the default route
                # takes sigma on the special-function unit
                gdpa.gdpa_set_act_route(gdpa.GDPA_ROUTE_ALU)
                try:
                    r = measure_forward(name, args, rank, world, local, dist, gdpa, with_e2e=False)
                finally:
                    gdpa.gdpa_set_act_route(gdpa.GDPA_ROUTE_SFU)
                others[name]["alu_route"] = {"ms_per_step": r["ms_per_step"], "value": r["value"],
                                             "roofline_frac": r["roofline"]["frac"],
                                             "launch_ms": r["roofline"]["launch_ms"]}
                del r

    per_rank = head["per_rank_flops"]
    skew = max(per_rank) / (sum(per_rank) / len(per_rank)) if sum(per_rank) > 0 else 1.0
    if rank == 0:
        line = {
            "metric": METRIC, "value": head["value"], "unit": "TFLOPS", "n_gpus": world, "steps": K,
            "warmup": max(3, args.warmup), "ms_per_step": head["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "mxfp8 (Q, K, V, P) + bf16 O" if w.mx else "bf16",
            "data": "synthetic",
            "config": {"workload": "%s: %s" % (args.workload, RECIPES[args.workload]), "seed": w.seed,
                       "global_batch": w.B * world, "tokens_q": Tq, "tokens_kv": head["Tkv"],
                       "l2": "inputs %.2f GB > 126 MB L2; no flush" % head["input_gb"],
                       "parallelism": ("dp%d: LPT shard of one seeded batch of %d sequences, whole sequences per "
                                       "rank, no collective; useful-FLOP skew max/mean %.4f"
                                       % (world, w.B * world, skew)) if world > 1 else "dp1",
                       "entry": ("gdpa_fwd_mxfp8" if w.mx else "gdpa_fwd_async")
                                + " (host plan + upload + kernel per step)"},
            "clocks": head["clocks"],
            "e2e": head["e2e"],
            "gpu_launches": K,
            "roofline": head["roofline"],
            "cpu_baseline": cpu,
        }
        if others:
            line["workloads"] = others
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def backward_bytes(batch) -> float:
    """Read Q, K, V, O, dO once, write dq, dk, dv once (bf16), plus the fp32 lse."""
    Tq, Tkv = int(batch.q_offsets[-1]), int(batch.kv_offsets[-1])
    return 2.0 * batch.H * batch.D * (4 * Tq + 4 * Tkv) + 4.0 * batch.H * Tq


def run_backward(args, rank, world, local):
    import torch

    from jagged_attention_recommender_gb300 import build as gbuild
    from jagged_attention_recommender_gb300 import gdpa

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    gbuild.build()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    w = WORKLOADS[args.workload]
    batch, per_rank = bench_batch(args.workload, rank, world)
    flops = 2.5 * useful_flops(batch)
    nbytes = backward_bytes(batch)
    H, D, B = w.H, w.D, batch.B
    Tq, Tkv = int(batch.q_offsets[-1]), int(batch.kv_offsets[-1])

    def dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()

    q, k, v = dev(batch.q), dev(batch.k), dev(batch.v)
    g = torch.Generator(device="cuda").manual_seed(w.seed + 17)
    dout = torch.randn((Tq, H, D), device="cuda", generator=g).to(torch.bfloat16)
    qo = torch.from_numpy(batch.q_offsets).cuda()
    ko = torch.from_numpy(batch.kv_offsets).cuda()
    out = torch.empty((Tq, H, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((Tq, H), dtype=torch.float32, device="cuda")
    dq = torch.empty_like(out)
    dk = torch.empty((Tkv, H, D), dtype=torch.bfloat16, device="cuda")
    dv = torch.empty_like(dk)
    h_qo, h_ko = batch.q_offsets, batch.kv_offsets
    stream = torch.cuda.current_stream()
    if w.window_blocks < 0:  # sliding window of -window_blocks tokens
        gdpa.gdpa_fwd_sliding(q, k, v, h_qo, h_ko, qo, ko, B, H, D, w.act, -w.window_blocks, w.scale, out, lse, stream)
    else:
        gdpa.gdpa_fwd_lse(q, k, v, h_qo, h_ko, qo, ko, B, H, D, w.act, w.window_blocks, w.scale, out, lse, stream)

    def step():
        if w.window_blocks < 0:
            gdpa.gdpa_bwd_sliding(q, k, v, out, dout, lse, h_qo, h_ko, qo, ko, B, H, D, w.act, -w.window_blocks,
                                  w.scale, dq, dk, dv, stream)
        else:
            gdpa.gdpa_bwd(q, k, v, out, dout, lse, h_qo, h_ko, qo, ko, B, H, D, w.act, w.window_blocks, w.scale, dq,
                          dk, dv, stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    st = gdpa.gdpa_device_status()
    if st != gdpa.GDPA_OK:
        raise SystemExit("device status after warm-up: " + gdpa.gdpa_status_string(st))
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                           else int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local]))
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    e0.record(stream)
    for i in range(K):
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    st = gdpa.gdpa_device_status()
    if st != gdpa.GDPA_OK:
        raise SystemExit("device status after timing: " + gdpa.gdpa_status_string(st))
    elapsed_ms = e0.elapsed_time(e1)
    launch_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    if dist:
        t = torch.tensor([elapsed_ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed_ms = float(t.item())
    value = 2.5 * sum(per_rank) * K / (elapsed_ms / 1e3) / 1e12
    peaks, peak_src = load_peaks()
    bound = BOUND[args.workload]
    if bound == "tensor":
        achieved, peak, unit = flops / (launch_ms / 1e3) / 1e12, peaks["bf16_tflops"], "TFLOP/s"
    else:
        achieved, peak, unit = nbytes / (launch_ms / 1e3) / 1e9, peaks["hbm_gbs"], "GB/s"
    roofline = {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
                "traffic": None, "peak_source": peak_src + (" (burst)" if bound == "tensor" else ""),
                "launch_ms": launch_ms, "useful_flops_per_launch": flops, "algorithmic_bytes_per_launch": nbytes,
                "kernel": "gdpa_bwd step (prep + dq + dkdv kernels)"}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle

        rng = np.random.default_rng(2024)
        order = [int(s_) for s_ in rng.permutation(B)]
        do_bits = dout.view(torch.int16).cpu().numpy().view(np.uint16)

        def dout_of(seqs):
            return np.concatenate([do_bits[batch.q_offsets[s_]:batch.q_offsets[s_ + 1]] for s_ in seqs])

        # calibrate on one sequence (at most H threads busy), then time one
        # call over a sample sized for about --cpu-seconds on every core
        probe = batch.subset(order[:1])
        t0 = time.perf_counter()
        oracle.gdpa_bwd_batch(probe, dout_of(order[:1]))
        rate = useful_flops(probe) / max(time.perf_counter() - t0, 1e-3)
        rate *= max(1.0, min(oracle.num_cpus(), 4 * H) / H)
        seqs, acc = [], 0.0
        for s_ in order:
            seqs.append(s_)
            acc += useful_flops(batch.subset([s_]))
            if acc >= rate * args.cpu_seconds:
                break
        sub = batch.subset(seqs)
        t0 = time.perf_counter()
        oracle.gdpa_bwd_batch(sub, dout_of(seqs))
        spent = time.perf_counter() - t0
        cpu = {"value": 2.5 * useful_flops(sub) / spent / 1e12, "unit": "TFLOPS", "cores": oracle.num_cpus(),
               "kind": "oracle", "sample": "%d of %d sequences (seeded), all %d heads, %.1f s" % (
                   len(seqs), B, H, spent)}
    if rank == 0:
        line = {
            "metric": METRIC_BWD, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": K,
            "warmup": max(3, args.warmup), "ms_per_step": elapsed_ms / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "%s: %s" % (args.workload, RECIPES[args.workload]), "seed": w.seed,
                       "pass": "backward", "global_batch": w.B * world, "tokens_q": Tq, "tokens_kv": Tkv,
                       "l2": "inputs %.2f GB > 126 MB L2; no flush" % (
                           (q.numel() + k.numel() + v.numel() + out.numel() + dout.numel()) * 2 / 1e9),
                       "parallelism": ("dp%d: LPT shard of one seeded batch of %d sequences, no collective"
                                       % (world, w.B * world)) if world > 1 else "dp1",
                       "entry": "gdpa_bwd (host work lists + upload + 3 kernels per step)"},
            "clocks": clocks,
            "e2e": None,
            "gpu_launches": 3 * K,
            "roofline": roofline,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def main():
    args = parse_args()
    rank, world, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.pass_ == "backward":
        return run_backward(args, rank, world, local)
    return run_ours(args, rank, world, local)


if __name__ == "__main__":
    sys.exit(main())
