#!/usr/bin/env python
"""Benchmark of the bucketed N-replica gradient average on GB300.

Headline workload (one "step" = one pass of the gradient-sync hot path):
ResNet-50 parameter layout (161 tensors, 25,557,032 fp32 elements), 8
replicas' gradients resident in HBM, planned into 25 MiB buckets in reverse
registration order (5 buckets), each bucket averaged by one
ddp_bucket_allreduce_mean launch.  The step's 5 per-bucket launches are
captured once into a CUDA Graph on a side stream, so a step's host dispatch
is one graph launch; the timed region replays it K times.

Metric: algorithmic HBM bytes moved per second, (N+1)*4 bytes per element
(N replica reads + one fp32 write), and that rate as a fraction of the
measured HBM copy bandwidth.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs under torchrun: every rank runs its own copy of the workload on its
own GPU (replicas only — the single-GPU path has no cross-GPU exchange), the
timed region is bracketed by barriers, and the slowest rank's time is used.
--impl reference times the CPU oracle (the plain numpy definition) on the host
cores instead, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import datetime as _dt
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

MiB = 1 << 20
N_REPLICAS = 8
CAP_BYTES = 25 * MiB
METRIC = "bucket allreduce-mean GB/s (HBM bytes moved) & % of HBM roofline, 1×GB300"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 10 ** 6
# Sampler roofline (integer arithmetic; the 8 bytes written per index are far below HBM's rate).
# One encryption of the keyed permutation is 4 Feistel rounds, each the MurmurHash3 32-bit
# finalizer of (half xor round key) masked and xored into the other half: 2 multiplies, 3 shifts
# and 6 logic operations; the cycle walk then composes the value (1 multiply-add) and compares it
# with n (1): 46 integer operations per encryption.  Cycle walking takes 2^bits / n encryptions per
# index on average (bits = ceil(log2 n): the domain over the values in range).  An SM has two
# integer-capable pipes of 64 lanes per cycle each: the ALU (logic operations, compares, shifts)
# and the FMA-heavy pipe (multiplies, multiply-adds, and shifts written as multiply-highs).  The
# 25 logic operations and compares can issue only on the ALU and the 9 multiplies only on the
# other pipe; the 12 shifts can go to either, so the best split puts them all on the FMA-heavy
# pipe (21 operations there) and the ALU's 25 set the pace: max(25, 46 / 2) / 64 SM cycles per
# encryption.
SAMPLER_OPS_PER_ENCRYPTION = 4 * (2 + 3 + 6) + 2
SAMPLER_ALU_ONLY_OPS = 4 * 6 + 1
SAMPLER_PIPE_LANES = 64
GB300_SMS = 152
STEP_STREAMS = 8       # streams the headline step's bucket launches are spread over
SYNCBN_CALLS = 12      # calls captured per graph in the SyncBN rows (a multiple of every input-set count)
SAMPLER_CALLS = 20     # calls (epochs 1..20) captured per graph in the sampler row


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=4000)
    p.add_argument("--warmup", type=int, default=200)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--e2e-steps", type=int, default=5)
    p.add_argument("--no-rows", action="store_true", help="skip the SGD / SyncBN / sampler rows")
    p.add_argument("--rows", default=None,
                   help="comma-separated subset of the side-row groups to run: linear (the Linear(128,10) step's "
                        "latency), gpt2 (SGD, SGD with the bf16 copy, bf16 average), accum (accumulation, clipped step), orders (ring and tree order), syncbn, "
                        "sampler, sweep; default all")
    p.add_argument("--rows-out", default=None, help="also append every side-row line to this file")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU work budget of the oracle baseline")
    return p.parse_args()


# ----------------------------------------------------------------------------- environment

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_max(value: float, world: int, device=None) -> float:
    """The largest of every rank's `value` (all ranks get it).  The tensor
    lives on `device`: a CUDA device for NCCL, the CPU for gloo."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_rate(world: int, bytes_per_rank_step: float, steps: int, max_elapsed_ms: float) -> float:
    """Whole-job GB/s: every rank moved bytes_per_rank_step per step; the
    job took as long as its slowest rank."""
    return world * bytes_per_rank_step * steps / (max_elapsed_ms * 1e-3) / 1e9


def load_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clock, power and throttle reasons while a
    region runs; samples are kept with their host timestamps."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return []
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append({"t": ts, "sm": float(parts[2]), "sm_max": float(parts[3]),
                             "power": float(parts[4]) if parts[4] not in ("[N/A]", "N/A") else None,
                             "hw_slowdown": parts[6], "hw_thermal": parts[7], "sw_thermal": parts[8],
                             "sw_power_cap": parts[9]})
            except ValueError:
                continue
        return rows


def summarize_clocks(rows, t0, t1):
    inside = [r for r in rows if t0 <= r["t"] <= t1]
    window = "timed region"
    if not inside:       # region shorter than the sampling period: nearest samples around it
        inside = sorted(rows, key=lambda r: min(abs(r["t"] - t0), abs(r["t"] - t1)))[:3]
        window = "nearest samples to a short timed region"
    if not inside:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": "no samples"}
    reasons = set()
    for r in inside:
        for key, name in (("hw_slowdown", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                          ("sw_thermal", "sw_thermal_slowdown"), ("sw_power_cap", "sw_power_cap")):
            if r[key].lower().startswith("active"):
                reasons.add(name)
    pw = [r["power"] for r in inside if r["power"] is not None]
    return {"sm_mhz": statistics.median(r["sm"] for r in inside), "sm_max_mhz": max(r["sm_max"] for r in inside),
            "reasons": sorted(reasons), "samples": len(inside), "window": window,
            "power_w_max": max(pw) if pw else None}


def profile_traffic(source_files, elems_per_launch):
    """ncu DRAM bytes per launch of the dominant kernel: the committed
    summary's bytes per element (measured on one launch of the same kernel)
    times the elements of an average launch here, or None if the kernel's
    sources no longer hash to what was profiled."""
    path = os.path.join(ROOT, "profiles", "mean_kernel_resnet50.md")
    try:
        txt = open(path, encoding="utf-8").read()
    except OSError:
        return None, None
    m = re.search(r"traffic_bytes_per_element:\s*([0-9.eE+]+)\s+source_sha256:\s*([0-9a-f]+)", txt)
    if not m:
        return None, None
    h = hashlib.sha256()
    for f in source_files:
        with open(f, "rb") as fh:
            h.update(fh.read())
    if h.hexdigest()[:16] != m.group(2)[:16]:
        return None, "kernel changed since the ncu capture"
    return float(m.group(1)) * elems_per_launch, None


def kernel_source_hash():
    csrc = os.path.join(ROOT, "gradient_sync_ddp_gb300", "csrc")
    return [os.path.join(csrc, f) for f in ("allreduce.cu", "common.cuh", "host_common.h")]


# ----------------------------------------------------------------------------- workload

def resnet50_plan(plan_fn):
    import workloads
    num = workloads.numels(workloads.resnet50_layout())
    return num, plan_fn(num, 4, CAP_BYTES)


def algorithmic_bytes(plan, n=N_REPLICAS):
    return sum((n + 1) * 4 * b[1] for b in plan["buckets"])


def cpu_oracle_rate(plan, budget_s: float, seed_base: int = 0):
    """Time the oracle's rank-ordered average on the host over a bounded
    sample of the workload: the first k elements of every bucket, k chosen
    so that the timed passes take about budget_s seconds."""
    import numpy as np

    import oracle
    gen = np.random.Generator(np.random.PCG64(1234 + 200 + seed_base))
    probe = 1 << 18
    reps = [(gen.standard_normal(probe, dtype=np.float32) * np.float32(0.01)) for _ in range(N_REPLICAS)]
    t = time.perf_counter()
    oracle.grad_mean(reps)
    per_elem = max((time.perf_counter() - t) / probe, 1e-10)
    full = max(b[1] for b in plan["buckets"])
    k = int(min(full, max(probe, budget_s / per_elem / len(plan["buckets"]) / 3)))
    data = [[(gen.standard_normal(min(k, b[1]), dtype=np.float32) * np.float32(0.01)) for _ in range(N_REPLICAS)]
            for b in plan["buckets"]]
    elems = sum(len(d[0]) for d in data)
    passes = 0
    t0 = time.perf_counter()
    while True:
        for d in data:
            oracle.grad_mean(d)
        passes += 1
        if time.perf_counter() - t0 >= budget_s or passes >= 1000:
            break
    dt = time.perf_counter() - t0
    nbytes = (N_REPLICAS + 1) * 4 * elems * passes
    line = {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"first {k:,} elements of each of the {len(plan['buckets'])} buckets x {N_REPLICAS} "
                      f"replicas ({elems:,} elements per pass), {passes} passes in {dt:.1f} s, numpy "
                      f"single-threaded on {os.cpu_count()} host cores"}
    line["c_oracle"] = c_oracle_rates(data)
    return line


def c_oracle_rates(data, budget_s: float = 3.0):
    """Context beside the numpy figure: the plain-C restatement of the same
    average (oracle/mean_ref.c, pinned bit-exact to the numpy oracle) on the
    same sample, single-threaded and split over the host's threads."""
    from oracle import cref
    if not cref.available():
        return None
    out = {}
    elems = sum(len(d[0]) for d in data)
    for name, threaded in (("single_thread", False), ("threads", True)):
        passes, t0 = 0, time.perf_counter()
        while True:
            for d in data:
                cref.grad_mean_c(d, threaded=threaded)
            passes += 1
            if time.perf_counter() - t0 >= budget_s or passes >= 1000:
                break
        dt = time.perf_counter() - t0
        out[name + "_GBps"] = (N_REPLICAS + 1) * 4 * elems * passes / dt / 1e9
    out["threads"] = cref.threads()
    return out


# ----------------------------------------------------------------------------- reference arm

def run_reference(args, world, rank):
    if rank != 0:
        return
    sys.path.insert(0, ROOT)
    import numpy as np

    import oracle
    import workloads
    num, plan = resnet50_plan(oracle.plan_buckets)
    nb = len(plan["buckets"])
    gen = np.random.Generator(np.random.PCG64(1234 + 200))
    probe = 1 << 18
    reps = [(gen.standard_normal(probe, dtype=np.float32) * np.float32(0.01)) for _ in range(N_REPLICAS)]
    t = time.perf_counter()
    oracle.grad_mean(reps)
    per_elem = max((time.perf_counter() - t) / probe, 1e-10)
    budget = 120.0 / max(1, args.steps + args.warmup)          # whole run: about two minutes
    k = int(min(max(b[1] for b in plan["buckets"]), max(4096, budget / per_elem / nb)))
    data = [[workloads.normal_f32(workloads.rng(2, r), min(k, b[1]), 0.0, 0.01) for r in range(N_REPLICAS)]
            for b in plan["buckets"]]
    elems = sum(len(d[0]) for d in data)
    for _ in range(args.warmup):
        for d in data:
            oracle.grad_mean(d)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        for d in data:
            oracle.grad_mean(d)
    dt = time.perf_counter() - t0
    value = (N_REPLICAS + 1) * 4 * elems * args.steps / dt / 1e9
    sample = (f"each step: first {k:,} elements of each of the {nb} buckets x {N_REPLICAS} replicas "
              f"({elems:,} elements), numpy single-threaded")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / max(1, args.steps) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic: seeded N(0, 0.01) fp32 replica gradients (numpy PCG64)",
            "config": workload_config(plan, num),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config(plan, num):
    return {"workload": "ResNet-50 parameter layout (161 tensors, 25,557,032 fp32 elements), 8 replicas, "
                        "25 MiB buckets in reverse registration order, rank-ordered mean",
            "replicas": N_REPLICAS, "tensors": len(num), "elements": sum(num), "buckets": len(plan["buckets"]),
            "bucket_cap_mib": 25, "bytes_per_step": algorithmic_bytes(plan),
            "l2": "inputs larger than L2 (818 MB of replica gradients read per step vs 129 MB L2); no flush",
            "parallelism": "replicas only: each GPU averages its own 8 resident replicas"}


# ----------------------------------------------------------------------------- our arm

def run_ours(args, world, rank, local):
    import torch
    import torch.distributed as dist

    import workloads
    import __graft_entry__
    __graft_entry__.build()
    import gradient_sync_ddp_gb300 as g

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl")

    num, plan = resnet50_plan(g.ddp_plan_buckets)
    total = plan["total_elems"]
    buckets = plan["buckets"]
    reps = [workloads.device_normal((total,), 0.0, 0.01, workloads.seed_for(2, r) + 1000 * rank, device=dev)
            for r in range(N_REPLICAS)]
    out = torch.empty(total, device=dev)
    side = torch.cuda.Stream(device=dev)

    def launch(b, stream=None):
        off, n = buckets[b][0], buckets[b][1]
        g.ddp_bucket_allreduce_mean([x[off:off + n] for x in reps], out[off:off + n], stream=stream)

    # One step = the bucket launches in bucket order.  The buckets are disjoint, so each goes out on its own
    # stream (a pool of up to STEP_STREAMS, forked from and joined back into the side stream): a bucket's
    # CTAs then start on the SMs the previous bucket's last CTAs free, instead of after its whole grid.
    bucket_streams = [torch.cuda.Stream() for _ in range(min(len(buckets), STEP_STREAMS))]

    def step_body():
        cur = torch.cuda.current_stream()
        for st in bucket_streams:
            st.wait_stream(cur)
        for b in range(len(buckets)):
            launch(b, bucket_streams[b % len(bucket_streams)])
        for st in bucket_streams:
            cur.wait_stream(st)

    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step_body()
    torch.cuda.synchronize()
    step_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(step_graph, stream=side):
        step_body()
    torch.cuda.synchronize()

    step_bytes = algorithmic_bytes(plan)
    nb = len(buckets)
    K, W = args.steps, args.warmup

    with torch.cuda.stream(side):
        for _ in range(W):
            step_graph.replay()
    torch.cuda.synchronize()

    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
        time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_host0 = time.time()
    with torch.cuda.stream(side):
        t_start.record()
        for _ in range(K):
            step_graph.replay()
        t_end.record()
    torch.cuda.synchronize()
    t_host1 = time.time()
    if world > 1:
        dist.barrier()
    clock_rows = sampler.stop() if rank == 0 else []
    local_ms = t_start.elapsed_time(t_end)
    elapsed_ms = dist_max(local_ms, world, dev)
    value = weak_scaling_rate(world, step_bytes, K, elapsed_ms)

    # The dominant kernel's own launch duration.  Inside the step the 5 launches overlap on their
    # streams, so the step time over 5 is not one launch's duration.  Here the same 5 launches run
    # one after another on the side stream (one graph, K replays between events on that stream):
    # each launch then has the GPU to itself, and the region time over the K x 5 launches is the
    # kernel's average launch duration.
    serial_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(serial_graph, stream=side):
        for b in range(nb):
            launch(b)
    with torch.cuda.stream(side):
        for _ in range(max(W, 3)):
            serial_graph.replay()
    torch.cuda.synchronize()
    k_start, k_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(side):
        k_start.record()
        for _ in range(K):
            serial_graph.replay()
        k_end.record()
    torch.cuda.synchronize()
    avg_launch_ms = k_start.elapsed_time(k_end) / (K * nb)
    achieved = (step_bytes / nb) / (avg_launch_ms * 1e-3) / 1e9
    peak, peak_kind = load_peak()
    traffic, traffic_note = profile_traffic(kernel_source_hash(), step_bytes / nb / ((N_REPLICAS + 1) * 4))

    # End to end through the public API, host buffers in and out, two ways:
    #  "copy":      every step copies the replicas from pinned host memory into HBM bucket by bucket on one
    #               copy stream, each bucket's average starts once its slices have arrived, and its result
    #               goes back to pinned host memory on a third stream (the copy of bucket b's result overlaps
    #               the inbound copies of the later buckets);
    #  "zero-copy": the same 5 bucket calls given the pinned host buffers themselves: the kernels read the
    #               replicas over NVLink-C2C (coherent host memory) and write the average to host memory.
    host_reps = [torch.empty(total, dtype=torch.float32, pin_memory=True) for _ in range(N_REPLICAS)]
    for h, d in zip(host_reps, reps):
        h.copy_(d)
    host_out = torch.empty(total, dtype=torch.float32, pin_memory=True)
    torch.cuda.synchronize()
    h2d_stream, k_stream, d2h_stream = (torch.cuda.Stream(device=dev) for _ in range(3))

    def launch_host(b):
        off, n = buckets[b][0], buckets[b][1]
        g.ddp_bucket_allreduce_mean([x[off:off + n] for x in host_reps], host_out[off:off + n])

    def e2e_copy_step():
        cur = torch.cuda.current_stream()
        for st in (h2d_stream, k_stream, d2h_stream):
            st.wait_stream(cur)
        for b in range(nb):
            off, n = buckets[b][0], buckets[b][1]
            with torch.cuda.stream(h2d_stream):
                for h, d in zip(host_reps, reps):
                    d[off:off + n].copy_(h[off:off + n], non_blocking=True)
            k_stream.wait_stream(h2d_stream)
            launch(b, k_stream)
            d2h_stream.wait_stream(k_stream)
            with torch.cuda.stream(d2h_stream):
                host_out[off:off + n].copy_(out[off:off + n], non_blocking=True)
        for st in (h2d_stream, k_stream, d2h_stream):
            cur.wait_stream(st)

    def e2e_zero_copy_step():
        for b in range(nb):
            launch_host(b)

    def time_e2e(fn):
        with torch.cuda.stream(side):
            fn()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(side):
            e0.record()
            for _ in range(args.e2e_steps):
                fn()
            e1.record()
        torch.cuda.synchronize()
        return weak_scaling_rate(world, step_bytes, args.e2e_steps, dist_max(e0.elapsed_time(e1), world, dev))

    e2e_copy = time_e2e(e2e_copy_step)
    copy_check = bool(torch.equal(host_out, out.cpu()))
    e2e_zero = time_e2e(e2e_zero_copy_step)

    # the host link on its own: copy-engine H2D of the replicas, for the bound the e2e figures sit under
    with torch.cuda.stream(side):
        l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        l0.record()
        for _ in range(3):
            for h, d in zip(host_reps, reps):
                d.copy_(h, non_blocking=True)
        l1.record()
    torch.cuda.synchronize()
    h2d_gbs = 3 * N_REPLICAS * total * 4 / (l0.elapsed_time(l1) * 1e-3) / 1e9
    host_check = copy_check and bool(torch.equal(host_out, out.cpu()))   # both modes computed the same average

    if rank == 0:
        # diagnostic row (not the headline): each bucket's launch timed on its own, eagerly
        per_bucket = []
        with torch.cuda.stream(side):
            for b in range(nb):
                ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                ea.record()
                for _ in range(20):
                    launch(b)
                eb.record()
                per_bucket.append((ea, eb))
        torch.cuda.synchronize()
        emit_row("headline_buckets", {
            "workload": "ResNet-50 step, each bucket's launch timed alone (20 eager launches each)",
            "bytes": [(N_REPLICAS + 1) * 4 * b[1] for b in buckets],
            "us": [ea.elapsed_time(eb) / 20 * 1e3 for ea, eb in per_bucket]}, args.rows_out)

    if rank == 0 and world == 1 and not args.no_rows:
        del host_reps, host_out
        only = None if args.rows is None else {r.strip() for r in args.rows.split(",") if r.strip()}
        bench_rows(g, torch, dev, peak, peak_kind, only, args.rows_out)

    if rank == 0:
        cpu = None if args.no_cpu_baseline or world > 1 else cpu_oracle_rate(plan, args.cpu_seconds)
        clocks = summarize_clocks(clock_rows, t_host0, t_host1)
        line = headline(value=value, world=world, K=K, W=W, elapsed_ms=elapsed_ms, plan=plan, num=num,
                        peak=peak, peak_kind=peak_kind, achieved=achieved, avg_launch_ms=avg_launch_ms,
                        traffic=traffic, traffic_note=traffic_note, cpu=cpu, e2e_copy=e2e_copy,
                        e2e_zero=e2e_zero, h2d_gbs=h2d_gbs, host_check=host_check,
                        e2e_steps=args.e2e_steps, clocks=clocks, step_streams=len(bucket_streams))
        emit_headline(line)
    if world > 1:
        dist.destroy_process_group()


HEADLINE_MAX_BYTES = 3500   # the result line stays short: the last line of stdout, read from its tail


def headline(*, value, world, K, W, elapsed_ms, plan, num, peak, peak_kind, achieved, avg_launch_ms, traffic,
             traffic_note, cpu, e2e_copy, e2e_zero, h2d_gbs, host_check, e2e_steps, clocks, step_streams):
    """The one result line of the run (a flat, short dict): the headline
    metric, the dominant kernel's roofline, the CPU oracle baseline, the
    end-to-end figure and the clocks of the timed region."""
    nb = len(plan["buckets"])
    step_bytes = algorithmic_bytes(plan)
    total = plan["total_elems"]
    cfg = workload_config(plan, num)
    cfg["schedule"] = f"one CUDA graph per step, each bucket launch on its own stream ({step_streams} streams)"
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": traffic, "peak_source": f"{peak_kind} HBM copy bandwidth",
            "kernel": "mean_kernel (fp32, rank order, N=8)",
            "algorithmic_bytes_per_launch": step_bytes / nb, "avg_launch_us": avg_launch_ms * 1e3,
            "launch_timing": "the step's 5 launches serialised on one stream, K graph replays, CUDA events"}
    if traffic_note:
        roof["traffic_note"] = traffic_note
    if cpu is not None:
        cpu = {k: v for k, v in cpu.items() if k != "c_oracle"}
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": elapsed_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic: seeded N(0, 0.01) fp32 replica gradients drawn on the device",
        "config": cfg,
        "hbm_fraction": value / world / peak,
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_copy, "unit": "GB/s", "h2d_bytes_per_step": N_REPLICAS * total * 4,
                "d2h_bytes_per_step": total * 4, "steps": e2e_steps, "mode": "copy (pinned host <-> HBM, "
                "pipelined by bucket)", "zero_copy_mode_value": e2e_zero, "modes_agree_bitwise": host_check,
                "host_link_h2d_GBps": h2d_gbs},
        "gpu_launches": K * nb,
        "clocks": clocks,
    }
    return line


def emit_row(name, row, path=None):
    """One side measurement as its own JSON line on stdout (and appended to
    `path` if given), printed before the result line."""
    rec = {"row": name, **row}
    s = json.dumps(rec)
    print(s, flush=True)
    if path:
        with open(path, "a", encoding="utf-8") as f:
            f.write(s + "\n")


def emit_headline(line):
    """Print the result line: the last line of stdout, compact."""
    s = json.dumps(line, separators=(",", ":"))
    if len(s) > HEADLINE_MAX_BYTES:
        raise RuntimeError(f"result line is {len(s)} bytes, over {HEADLINE_MAX_BYTES}")
    sys.stdout.flush()
    print(s, flush=True)


def _time_launches(torch, fn, iters, stream):
    """Mean device time (ms) of one fn() call: fn's launches are captured once
    into a CUDA Graph on `stream` (after 3 eager warm-up calls) and the graph
    is replayed 3 times untimed, then `iters` times between two events, so
    host dispatch cost is not part of the figure."""
    with torch.cuda.stream(stream):
        for _ in range(3):
            fn()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        fn()
    with torch.cuda.stream(stream):
        for _ in range(3):
            graph.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record()
        for _ in range(iters):
            graph.replay()
        b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / iters


def _fan_out(torch, calls, streams):
    """Run calls[i] on streams[i % len(streams)], forked from and joined back
    into the current stream (independent buckets overlap; capturable)."""
    cur = torch.cuda.current_stream()
    for st in streams:
        st.wait_stream(cur)
    for i, call in enumerate(calls):
        with torch.cuda.stream(streams[i % len(streams)]):
            call()
    for st in streams:
        cur.wait_stream(st)


def bench_rows(g, torch, dev, peak, peak_kind, only=None, rows_out=None):
    """The other rows of the hot path, each on its own workload (not part of
    the headline value): fused SGD on GPT-2 small, SyncBN on the four
    activation shapes, the ImageNet-size sampler, and the bf16 average.
    Each row is printed as its own JSON line (emit_row) as soon as it is
    measured."""
    import workloads
    side = torch.cuda.Stream(device=dev)
    pool = [torch.cuda.Stream(device=dev) for _ in range(2)]   # the two GPT-2 buckets are disjoint

    def want(group):
        return only is None or group in only

    layout, first = workloads.gpt2_small_layout()      # GPT-2 small parameter list (gpt2 and accum rows)
    num = workloads.numels(layout)

    if want("linear"):
        # Linear(128,10): 4 fp32 replicas of 1,290 gradient elements, average + SGD lr 0.1 (no momentum) in one
        # launch; 31 KB per step, so the figure is the call's latency (20 calls per graph replay)
        numel_l = sum(workloads.numels(workloads.linear_128_10_layout()))   # 1,290
        reps_l = [workloads.device_normal((numel_l,), 0.0, 1.0, workloads.seed_for(1, r), device=dev) for r in range(4)]
        theta_l = workloads.device_normal((numel_l,), 0.0, 0.1, workloads.seed_for(1, 99), device=dev)
        ms = _time_launches(torch, lambda: [g.ddp_bucket_allreduce_sgd(reps_l, theta_l, None, 0.1, 0.0, 0.0)
                                            for _ in range(20)], 10, side) / 20
        nbytes = (4 * 4 + 8) * numel_l
        emit_row("sgd_linear_128_10", {"workload": "Linear(128,10), 4 fp32 replicas (1,290 elements), average + SGD "
                                                 "lr 0.1 in one launch", "ms": ms, "us": ms * 1e3, "bytes": nbytes,
                                     "GBps": nbytes / ms / 1e6, "frac": None, "launches": 1,
                                     "note": "latency-bound (31 KB per call): the figure is µs per call",
                                     "calls_per_graph": 20}, rows_out)
        del reps_l, theta_l

    if want("gpt2"):
        # fused SGD, GPT-2 small DEEP/FIRST, bf16 grads, momentum 0.9, wd 1e-4
        plan = g.ddp_plan_buckets(num, 2, 0, g.PLAN_DEEP_FIRST, first)
        total = plan["total_elems"]
        reps = [workloads.device_normal((total,), 0.0, 0.01, workloads.seed_for(3, r), device=dev,
                                        dtype=torch.bfloat16) for r in range(N_REPLICAS)]
        theta = workloads.device_normal((total,), 0.0, 0.02, workloads.seed_for(3, 99), device=dev)
        buf = torch.zeros(total, device=dev)

        def sgd_step():
            _fan_out(torch, [lambda off=off, n=n: g.ddp_bucket_allreduce_sgd(
                [x[off:off + n] for x in reps], theta[off:off + n], buf[off:off + n], 0.1, 0.9, 1e-4)
                for off, n, _, _ in plan["buckets"]], pool)
        ms = _time_launches(torch, sgd_step, 50, side)
        nbytes = sum((2 * N_REPLICAS + 16) * b[1] for b in plan["buckets"])
        emit_row("sgd_gpt2_small", {"workload": "GPT-2 small (124,439,808 params), 8 bf16 replicas, DEEP/FIRST buckets, "
                                              "SGD momentum 0.9 wd 1e-4", "ms": ms, "bytes": nbytes,
                                  "GBps": nbytes / ms / 1e6, "frac": nbytes / ms / 1e6 / peak, "launches": 2}, rows_out)

        # the same step also writing the bf16 compute copy of θ
        low = torch.empty(total, dtype=torch.bfloat16, device=dev)

        def sgd_cast_step():
            _fan_out(torch, [lambda off=off, n=n: g.ddp_bucket_allreduce_sgd_cast(
                [x[off:off + n] for x in reps], theta[off:off + n], buf[off:off + n], 0.1, 0.9, 1e-4, low[off:off + n])
                for off, n, _, _ in plan["buckets"]], pool)
        ms = _time_launches(torch, sgd_cast_step, 50, side)
        nbytes = sum((2 * N_REPLICAS + 18) * b[1] for b in plan["buckets"])
        emit_row("sgd_cast_gpt2_small", {"workload": "GPT-2 small, 8 bf16 replicas, SGD momentum 0.9 wd 1e-4 plus the "
                                                   "bf16 copy of θ", "ms": ms, "bytes": nbytes,
                                       "GBps": nbytes / ms / 1e6, "frac": nbytes / ms / 1e6 / peak, "launches": 2}, rows_out)
        del low

        # bf16 -> fp32 average of the same buckets
        outb = torch.empty(total, device=dev)

        def mean_bf16():
            _fan_out(torch, [lambda off=off, n=n: g.ddp_bucket_allreduce_mean([x[off:off + n] for x in reps],
                                                                              outb[off:off + n])
                             for off, n, _, _ in plan["buckets"]], pool)
        ms = _time_launches(torch, mean_bf16, 50, side)
        nbytes = sum((2 * N_REPLICAS + 4) * b[1] for b in plan["buckets"])
        emit_row("mean_bf16_gpt2_small", {"workload": "GPT-2 small, 8 bf16 replicas, DEEP/FIRST, average to fp32",
                                        "ms": ms, "bytes": nbytes, "GBps": nbytes / ms / 1e6,
                                        "frac": nbytes / ms / 1e6 / peak, "launches": 2}, rows_out)
        del reps, theta, buf, outb

    if want("accum"):
        # gradient accumulation (no_sync micro-step) and the clipped final step, GPT-2 small, fp32 accumulators
        plan4 = g.ddp_plan_buckets(num, 4, 0, g.PLAN_DEEP_FIRST, first)
        total4 = plan4["total_elems"]
        acc = [torch.zeros(total4, device=dev) for _ in range(N_REPLICAS)]
        micro = [workloads.device_normal((total4,), 0.0, 0.01, workloads.seed_for(3, r) + 50, device=dev,
                                         dtype=torch.bfloat16) for r in range(N_REPLICAS)]
        ms = _time_launches(torch, lambda: g.ddp_bucket_accumulate(micro, acc), 20, side)
        nbytes = (2 + 8) * N_REPLICAS * total4
        emit_row("accumulate_gpt2_small", {"workload": "GPT-2 small, 8 replicas, bf16 micro-step gradient added into "
                                                     "fp32 accumulators (no_sync)", "ms": ms, "bytes": nbytes,
                                         "GBps": nbytes / ms / 1e6, "frac": nbytes / ms / 1e6 / peak, "launches": 1}, rows_out)
        del micro
        gavg = torch.empty(total4, device=dev)
        theta = workloads.device_normal((total4,), 0.0, 0.02, workloads.seed_for(3, 99), device=dev)
        buf = torch.zeros(total4, device=dev)
        ws = torch.empty(g.ddp_norm_workspace_bytes(len(plan4["buckets"])), dtype=torch.uint8, device=dev)
        coef = torch.empty(1, device=dev)

        def clipped_step():
            _fan_out(torch, [lambda b=b, off=off, n=n: g.ddp_bucket_allreduce_mean_norm(
                [x[off:off + n] for x in acc], gavg[off:off + n], ws, b)
                for b, (off, n, _, _) in enumerate(plan4["buckets"])], pool)
            g.ddp_grad_norm_finalize(ws, len(plan4["buckets"]), 1.0, None, coef, None)
            _fan_out(torch, [lambda off=off, n=n: g.ddp_bucket_sgd(
                gavg[off:off + n], theta[off:off + n], buf[off:off + n], 0.1, 0.9, 1e-4, grad_scale=coef)
                for off, n, _, _ in plan4["buckets"]], pool)
        ms = _time_launches(torch, clipped_step, 20, side)
        nbytes = sum(((N_REPLICAS + 1) * 4 + 20) * b[1] for b in plan4["buckets"])
        emit_row("clipped_step_gpt2_small", {"workload": "GPT-2 small, 8 fp32 accumulated replicas: average with norm "
                                                       "side output, clip to 1.0, SGD momentum 0.9 wd 1e-4",
                                           "ms": ms, "bytes": nbytes, "GBps": nbytes / ms / 1e6,
                                           "frac": nbytes / ms / 1e6 / peak, "launches": 5}, rows_out)
        del acc, gavg, theta, buf

    if want("orders"):
        # the ResNet-50 step in the other reduction orders (ring chunks, pairwise tree), same schedule
        num_r = workloads.numels(workloads.resnet50_layout())
        plan_r = g.ddp_plan_buckets(num_r, 4, 25 << 20)
        reps_r = [workloads.device_normal((plan_r["total_elems"],), 0.0, 0.01, workloads.seed_for(2, r), device=dev)
                  for r in range(N_REPLICAS)]
        out_r = torch.empty(plan_r["total_elems"], device=dev)
        pool_r = [torch.cuda.Stream(device=dev) for _ in range(len(plan_r["buckets"]))]
        nbytes = sum((N_REPLICAS + 1) * 4 * b[1] for b in plan_r["buckets"])
        for name, flag in (("ring", g.FLAG_RING_ORDER), ("tree", g.FLAG_TREE_ORDER)):
            def ordered(flag=flag):
                _fan_out(torch, [lambda off=off, n=n: g.ddp_bucket_allreduce_mean(
                    [x[off:off + n] for x in reps_r], out_r[off:off + n], flags=flag)
                    for off, n, _, _ in plan_r["buckets"]], pool_r)
            ms = _time_launches(torch, ordered, 200, side)
            emit_row(f"mean_{name}_order_resnet50", {
                "workload": f"ResNet-50 step (5 x 25 MiB buckets, 8 fp32 replicas), {name}-order reduction",
                "ms": ms, "bytes": nbytes, "GBps": nbytes / ms / 1e6, "frac": nbytes / ms / 1e6 / peak,
                "launches": len(plan_r["buckets"])}, rows_out)
        del reps_r, out_r

    if want("syncbn"):
        # SyncBN, 4 shapes.  Calls cycle through R input sets (each set: 8 replicas' x and y) with
        # R·(x + y) >= 2.5 x L2, so a call never finds its x left in L2 by an earlier call: the stats
        # pass reads x from HBM.  (Within one call the apply's second read of x may still hit L2 when x
        # is smaller than L2; the bytes counted stay the algorithmic 6 per element.)
        for C, H, W in workloads.SYNCBN_SHAPES:
            B = workloads.SYNCBN_BATCH
            xbytes = 2 * N_REPLICAS * B * C * H * W
            R = max(1, -(-int(2.5 * L2_BYTES) // (2 * xbytes)))
            sets = []
            for k in range(R):
                xs = [workloads.device_normal((B, C, H, W), 0.5, 2.0, workloads.seed_for(4, r) + 100 * k, device=dev,
                                              dtype=torch.bfloat16) for r in range(N_REPLICAS)]
                sets.append((xs, [torch.empty_like(x) for x in xs]))
            ws = torch.empty(g.syncbn_workspace_bytes(N_REPLICAS, B, C, H, W), dtype=torch.uint8, device=dev)
            mean = torch.empty(C, device=dev)
            inv = torch.empty(C, device=dev)
            # SYNCBN_CALLS back-to-back calls per graph replay (as consecutive BN layers sit in a captured
            # step), so the figure is device time per call, not one graph launch's latency per call
            ms = _time_launches(torch, lambda: [g.syncbn_merge_apply(*sets[i % R], mean, inv, ws)
                                                for i in range(SYNCBN_CALLS)], 10, side) / SYNCBN_CALLS
            nbytes = 6 * N_REPLICAS * B * C * H * W
            parts = g.syncbn_channel_parts(N_REPLICAS, g.BF16, B, C, H, W)
            emit_row(f"syncbn_{C}x{H}x{W}", {"workload": f"SyncBN 8 x [32,{C},{H},{W}] bf16", "ms": ms, "bytes": nbytes,
                                           "GBps": nbytes / ms / 1e6, "frac": nbytes / ms / 1e6 / peak,
                                           "launches": 3 * parts, "streams": parts,
                                           "calls_per_graph": SYNCBN_CALLS, "input_sets": R,
                                           "l2": f"{R} input sets rotated: {R * 2 * xbytes / 1e6:.0f} MB of x and y "
                                                 f"against {L2_BYTES / 1e6:.0f} MB of L2"}, rows_out)
            del sets

    if want("sampler"):
        # sampler
        n, N = workloads.SAMPLER_N_ITEMS, workloads.SAMPLER_REPLICAS
        out = torch.empty(N * g.dist_sampler_num_samples(n, N, False), dtype=torch.int64, device=dev)
        ms = _time_launches(torch, lambda: [g.dist_sampler_indices(n, N, -1, 0, 1 + e, True, False, out)
                                            for e in range(SAMPLER_CALLS)], 10, side) / SAMPLER_CALLS
        # Integer roofline from the arithmetic (the ops of one encryption on the ALU and FMA-heavy
        # pipes), at the maximum SM clock
        bits = max(1, (n - 1).bit_length())
        enc_per_index = (1 << bits) / n
        sm_hz = 2.07e9
        pipe_ops = max(SAMPLER_ALU_ONLY_OPS, SAMPLER_OPS_PER_ENCRYPTION / 2)   # busiest pipe's ops per encryption
        peak_idx = GB300_SMS * SAMPLER_PIPE_LANES * sm_hz / (pipe_ops * enc_per_index)
        idx_per_s = out.numel() / (ms * 1e-3)
        emit_row("sampler_imagenet", {"workload": "1,281,167 items, 8 ranks, all ranks, shuffle", "ms": ms,
                                      "Mindex_per_s": idx_per_s / 1e6, "bytes": out.numel() * 8,
                                      "GBps": out.numel() * 8 / ms / 1e6, "bound": "alu",
                                      "peak_Mindex_per_s": peak_idx / 1e6, "frac": idx_per_s / peak_idx,
                                      "peak_basis": f"{SAMPLER_OPS_PER_ENCRYPTION} integer ops per encryption, "
                                                    f"{SAMPLER_ALU_ONLY_OPS} of them ALU-only, x "
                                                    f"{enc_per_index:.4f} encryptions per index; {GB300_SMS} SMs x "
                                                    f"{SAMPLER_PIPE_LANES} ALU lanes per cycle at 2070 MHz",
                                      "launches": 1, "calls_per_graph": SAMPLER_CALLS}, rows_out)
    if want("sweep"):
        # sweep (flat fp32 buffer split into cap-sized bucket launches, one graph per point): 1 KiB .. 1 GiB
        # per replica in x4 steps, N in {2, 4, 8, 16}, caps {1, 25, 100} MiB; a cap that does not change the
        # launch count is measured once; the 1 MiB split also as grouped launches (up to 1024 buckets each)
        for size in [1 << (10 + 2 * k) for k in range(11)]:
            numel = size // 4
            for n in (2, 4, 8, 16):
                reps = [workloads.device_normal((numel,), 0.0, 1.0, workloads.seed_for(5, r), device=dev)
                        for r in range(n)]
                outs = torch.empty(numel, device=dev)
                nbytes = (n + 1) * size
                l2 = "working set in L2" if nbytes < L2_BYTES else "larger than L2"
                iters = 200 if size <= (64 << 20) else 20
                seen = set()
                for cap in (1 << 20, 25 << 20, 100 << 20):
                    ce = cap // 4
                    nl = -(-numel // ce)
                    if nl in seen:
                        continue
                    seen.add(nl)

                    def flat_step(reps=reps, outs=outs, ce=ce, numel=numel):
                        for s0 in range(0, numel, ce):
                            e = min(numel, s0 + ce)
                            g.ddp_bucket_allreduce_mean([x[s0:e] for x in reps], outs[s0:e])
                    ms = _time_launches(torch, flat_step, iters, side)
                    emit_row("sweep_flat_fp32", {"bytes_per_replica": size, "replicas": n,
                                                 "cap_mib": cap >> 20 if nl > 1 else "any (one launch)",
                                                 "launches": nl, "us": ms * 1e3, "GBps": nbytes / ms / 1e6,
                                                 "frac": nbytes / ms / 1e6 / peak, "l2": l2}, rows_out)
                    if nl > 1 and cap == (1 << 20):
                        bl = [(s0, min(ce, numel - s0)) for s0 in range(0, numel, ce)]

                        def grouped(reps=reps, outs=outs, bl=bl):
                            for i in range(0, len(bl), 1024):
                                g.ddp_bucket_allreduce_mean_multi(reps, bl[i:i + 1024], outs)
                        ms = _time_launches(torch, grouped, iters, side)
                        emit_row("sweep_flat_fp32", {"bytes_per_replica": size, "replicas": n, "cap_mib": 1,
                                                     "launches": -(-len(bl) // 1024), "grouped": True,
                                                     "us": ms * 1e3, "GBps": nbytes / ms / 1e6,
                                                     "frac": nbytes / ms / 1e6 / peak, "l2": l2}, rows_out)
                del reps, outs
    emit_row("_peak", {"hbm_gbs": peak, "source": peak_kind}, rows_out)


def main():
    args = parse_args()
    world, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
