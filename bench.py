#!/usr/bin/env python
"""Throughput benchmark of the shifted-schedule sharded attention on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...      # the fp64 CPU oracle, timed

One step = one pass of the hot path over one batch of synthetic input: a
mercury_attn_sharded call on the Llama-3-8B-like GQA workload (B 1, 32 query /
8 KV heads, d 128, 32K tokens, causal, R = 8 virtual ranks, flat shift): it
shards Q and K/V, walks the shards in the shifted order, skips causally masked
shards, runs the tcgen05 attention patch and finalises O and LSE (the
per-step partials are combined on the fly, i.e. the log-sum-exp merge is
fused).  The separate partial + merge path is measured as a secondary figure
on the 2M-token MQA chunk (mercury_attn_partial + mercury_lse_merge), which is
where the merge's HBM bandwidth is reported.

Metric: attention TFLOP/s = 4 * d * (unmasked query/key pairs) * B * Hq per
step / time.  Inputs (384 MiB) are larger than L2, so no flush is needed
between steps.  Several GPUs (torchrun) run independent replicas: the path
needs no exchange on one GPU per replica, so value = sum of all ranks' work /
max-over-ranks time ("weak" scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from long_context_sharded_gb300.workloads import BENCH_WORKLOAD, WORKLOADS, attention_flops  # noqa: E402

METRIC = "attention TFLOP/s (bf16 fwd, 1×GB300) and % of dense BF16 peak; merge HBM GB/s"
UNIT = "TFLOP/s"
MERGE_WORKLOAD = "mqa_b1_hq8_hkv1_d128_sq2k_skv2m_r64_merge"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM traffic of one attention launch from an ncu capture (profiles/), valid
# only for the kernel source it was taken on (sha256 of attn_fwd.cu, first 16
# hex digits).  Reported as null once the kernel has changed.
ATTN_TRAFFIC = {"source_sha": "f5bee2595a63049d", "bytes_per_launch": 925422592,
                "profile": "profiles/attn_fwd_gqa32k_causal_full.md"}


# ------------------------------------------------------------------ helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Largest value of x over all ranks (identity on one rank)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_value(units_per_rank_per_step: float, steps: int, world: int, max_seconds: float) -> float:
    """Whole-job throughput: the work of all ranks over the slowest rank's time."""
    return units_per_rank_per_step * steps * world / max_seconds


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def source_sha(*paths: str) -> str:
    h = hashlib.sha256()
    for path in paths:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# the attention kernel's sources: its traffic record is valid for these bytes
ATTN_SOURCES = tuple(os.path.join(ROOT, "long_context_sharded_gb300", "csrc", f)
                     for f in ("attn_fwd.cu", "work.h", "ptx.cuh"))


class ClockSampler:
    """nvidia-smi samples (every 25 ms) of SM clock and throttle reasons."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        self.file = tempfile.TemporaryFile(mode="w+")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader", "-lms", "25"], stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return []
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.seek(0)
        rows = [line.strip().split(", ") for line in self.file if line.strip()]
        self.file.close()
        return rows

    @staticmethod
    def summarise(rows, t0, t1):
        """Median SM clock under load and the throttle reasons seen in [t0, t1]."""
        import datetime
        sm, sm_max, reasons = [], None, set()
        for r in rows:
            if len(r) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            if ts < t0 or ts > t1:
                continue
            try:
                sm.append(int(r[2].split()[0]))
                sm_max = int(r[3].split()[0])
            except (ValueError, IndexError):
                continue
            for name, val in zip(ClockSampler.REASONS, r[6:10]):
                if val.strip() == "Active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": sm_max,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ CPU oracle leg

def oracle_rate(q, k, v, w, seconds: float, seed: int):
    """Time the fp64 oracle on a bounded row sample of workload w.

    Returns (TFLOP/s, rows, seconds, sample description).  The flop count is
    the algorithmic 4*d per unmasked (q, k) pair of the sampled rows."""
    import numpy as np

    import oracle
    B, Hq, Sq, Skv, d, causal = w["B"], w["Hq"], w["Sq"], w["Skv"], w["d"], w["causal"]
    rng = np.random.default_rng(seed)
    off = Skv - Sq

    def pairs(rows):
        qi = rows % Sq
        return (np.minimum(qi + off + 1, Skv) if causal else np.full(rows.shape, Skv)).sum()

    n = 16
    while True:
        rows = np.sort(rng.choice(B * Hq * Sq, size=n, replace=False))
        t0 = time.perf_counter()
        oracle.attn(q, k, v, causal, rows=rows)
        dt = time.perf_counter() - t0
        if dt >= seconds or n >= B * Hq * Sq:
            break
        n = min(B * Hq * Sq, max(2 * n, int(n * seconds / max(dt, 1e-3) * 1.1)))
    flops = 4.0 * d * float(pairs(rows))
    return flops / dt / 1e12, n, dt, "%d seeded random query rows of %s (of %d)" % (n, w["name"], B * Hq * Sq)


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# --------------------------------------------------------------- GPU arm

def run_gpu(args):
    import torch

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    from long_context_sharded_gb300 import mercury as m
    from long_context_sharded_gb300.inputs import make_qkv

    w = dict(WORKLOADS[args.workload], name=args.workload)
    B, Hq, Hkv, Sq, Skv, d = w["B"], w["Hq"], w["Hkv"], w["Sq"], w["Skv"], w["d"]
    R, shift, causal = w["R"], w["shift"], w["causal"]
    partial = w["mode"] == "partial"
    flops = attention_flops(w)
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, d, seed=w["seed"], scale=w["scale"])
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    stream = torch.cuda.current_stream(dev)
    out = torch.empty((B, Hq, Sq, d), dtype=torch.float32, device=dev)
    lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=dev)
    o_part = lse_part = None
    if partial:
        o_part = torch.empty((R, B, Hq, Sq, d), dtype=torch.float32, device=dev)
        lse_part = torch.empty((R, B, Hq, Sq), dtype=torch.float32, device=dev)

    def step():
        if partial:
            m.mercury_attn_partial(qd, kd, vd, R, shift, causal, o_part, lse_part, stream)
            m.mercury_lse_merge(o_part, lse_part, out, lse, stream)
        else:
            m.mercury_attn_sharded(qd, kd, vd, R, shift, causal, out, lse, stream)

    launches_per_step = 2 if partial else 1
    for _ in range(args.warmup):
        step()
    m.mercury_sync_status(stream)

    sampler = ClockSampler(local)
    if rank == 0 and not args.no_clocks:
        sampler.start()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    barrier(world)
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    ev[0].record(stream)
    for i in range(args.steps):
        step()
        ev[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    barrier(world)
    rows = sampler.stop() if rank == 0 and not args.no_clocks else []
    m.mercury_sync_status(stream)
    per_step_ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    elapsed_s = ev[0].elapsed_time(ev[args.steps]) / 1e3
    max_s = max_over_ranks(elapsed_s, world, dev)
    value = aggregate_value(flops, args.steps, world, max_s) / 1e12

    # end to end through the public API with host buffers: every step copies
    # its inputs from pinned host memory to the device, runs the call and
    # copies O and LSE back.  Steps are pipelined the way a caller streaming
    # batches would: two device buffer slots, H2D on one stream, compute on
    # another, D2H on a third, so step i's copies overlap step i-1's compute.
    e2e = None
    if not args.no_e2e:
        qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
        slots = []
        for sidx in range(2):
            if sidx == 0:
                dq_, dk_, dv_, do_, dl_ = qd, kd, vd, out, lse
            else:
                dq_, dk_, dv_ = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
                do_, dl_ = torch.empty_like(out), torch.empty_like(lse)
            oh = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
            lh = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
            slots.append((dq_, dk_, dv_, do_, dl_, oh, lh))
        s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_cmp = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        e_steps = max(3, min(args.steps, 50))

        def e2e_step(i):
            dq_, dk_, dv_, do_, dl_, oh, lh = slots[i % 2]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_cmp[i % 2])      # slot's inputs no longer read
                dq_.copy_(qh, non_blocking=True)
                dk_.copy_(kh, non_blocking=True)
                dv_.copy_(vh, non_blocking=True)
                ev_in[i % 2].record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(ev_in[i % 2])
                if i >= 2:
                    s_cmp.wait_event(ev_out[i % 2])     # slot's outputs copied out
                if partial:
                    m.mercury_attn_partial(dq_, dk_, dv_, R, shift, causal, o_part, lse_part, s_cmp)
                    m.mercury_lse_merge(o_part, lse_part, do_, dl_, s_cmp)
                else:
                    m.mercury_attn_sharded(dq_, dk_, dv_, R, shift, causal, do_, dl_, s_cmp)
                ev_cmp[i % 2].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_cmp[i % 2])
                oh.copy_(do_, non_blocking=True)
                lh.copy_(dl_, non_blocking=True)
                ev_out[i % 2].record(s_out)

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        barrier(world)
        t0 = time.perf_counter()
        for i in range(e_steps):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        e_wall = time.perf_counter() - t0
        barrier(world)
        m.mercury_sync_status(s_cmp)
        e_s = max_over_ranks(e_wall, world, dev)
        h2d = sum(t.numel() * t.element_size() for t in (q, k, v))
        d2h = out.numel() * out.element_size() + lse.numel() * lse.element_size()
        e2e = {"value": round(aggregate_value(flops, e_steps, world, e_s) / 1e12, 3), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e_steps,
               "timing": "host wall clock around the steps, all streams synchronised at both ends",
               "pipelining": "2 buffer slots; H2D, compute and D2H on three streams"}
        del qh, kh, vh, slots

    peaks, peak_kind = load_peaks()
    launch_ms = statistics.mean(per_step_ms) if not partial else None
    roofline = None
    if not partial:
        achieved = flops / (launch_ms / 1e3) / 1e12
        traffic = (ATTN_TRAFFIC["bytes_per_launch"] if ATTN_TRAFFIC["source_sha"] == source_sha(*ATTN_SOURCES)
                   else None)
        roofline = {"kernel": "attn_fwd_kernel", "bound": "tensor", "achieved": round(achieved, 2),
                    "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                    "frac": round(achieved / peaks["bf16_tflops"], 4), "traffic": traffic,
                    "peak_kind": "%s burst bf16 (cuBLAS)" % peak_kind,
                    "frac_of_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4),
                    "algorithmic_flop_per_launch": flops,
                    "algorithmic_bytes_per_launch": (q.numel() + k.numel() + v.numel()) * 2
                    + out.numel() * 4 + lse.numel() * 4}

    secondary = None
    if not args.no_secondary and rank == 0 and world == 1:
        secondary = measure_merge_path(m, dev, stream, peaks, peak_kind)
        torch.cuda.empty_cache()
        # the schedule planner's estimates (built-in profile) beside the
        # measured times of the same schedules
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        prof = m.mercury_default_cost_profile(sms)
        top = m.mercury_plan_schedules(B, Hq, Hkv, Sq, Skv, d, causal, R, shift, 0, prof, 1)[0][0]
        cw = WORKLOADS[MERGE_WORKLOAD]
        ctop = m.mercury_plan_schedules(cw["B"], cw["Hq"], cw["Hkv"], cw["Sq"], cw["Skv"], cw["d"], cw["causal"],
                                        cw["R"], cw["shift"], 0, prof, 1)[0][0]
        secondary["schedule_model"] = {
            "bench_workload": {"schedule": [top.R, top.Rq, top.n_runs], "predicted_ms": round(top.predicted_us / 1e3, 4),
                               "measured_ms": round(statistics.median(per_step_ms), 4)},
            "merge_workload": {"schedule": [ctop.R, ctop.Rq, ctop.n_runs],
                               "predicted_ms": round(ctop.predicted_us / 1e3, 4),
                               "measured_ms_sharded_auto": secondary["sharded_auto_ms"]},
            "schedule_keys": ["R", "Rq", "n_runs"]}

    gemm = decode = None
    if not args.no_secondary and rank == 0 and world == 1:
        gemm = measure_gemm(m, dev, stream, peaks, peak_kind)
        torch.cuda.empty_cache()
        decode = measure_decode(m, dev, stream, peaks, peak_kind)
        torch.cuda.empty_cache()

    cpu = None
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        rate, n, dt, sample = oracle_rate(q, k, v, w, seconds=args.cpu_seconds, seed=w["seed"])
        cpu = {"value": round(rate, 6), "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
               "sample": sample, "seconds": round(dt, 2)}

    clocks = ClockSampler.summarise(rows, t_wall0, t_wall1) if rows else None
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(max_s * 1e3 / args.steps, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1)*%g, bf16)" % w["scale"],
            "config": {"workload": args.workload, "B": B, "Hq": Hq, "Hkv": Hkv, "Sq": Sq, "Skv": Skv,
                       "d": d, "R": R, "shift": shift, "causal": bool(causal),
                       "mode": "partial+merge" if partial else "fused",
                       "parallelism": "replicas" if world > 1 else "single GPU",
                       "l2": "inputs larger than L2 (%d MiB), no flush" % (
                           (q.numel() + k.numel() + v.numel()) * 2 >> 20)},
            "gpu_launches": args.steps * launches_per_step,
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
            "secondary": secondary, "gemm": gemm, "decode": decode,
            "per_step_ms": {"min": round(min(per_step_ms), 4), "median": round(statistics.median(per_step_ms), 4),
                            "max": round(max(per_step_ms), 4)},
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def measure_merge_path(m, dev, stream, peaks, peak_kind, reps: int = 10):
    """Partial + merge on the 2M-token MQA chunk: attention TFLOP/s of the
    partial kernel and HBM GB/s of the merge (bytes: every partial read once,
    the result written once)."""
    import torch

    from long_context_sharded_gb300.inputs import make_qkv
    w = WORKLOADS[MERGE_WORKLOAD]
    B, Hq, Hkv, Sq, Skv, d, R = w["B"], w["Hq"], w["Hkv"], w["Sq"], w["Skv"], w["d"], w["R"]
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, d, seed=w["seed"], scale=w["scale"])
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    del q, k, v
    op = torch.empty((R, B, Hq, Sq, d), dtype=torch.float32, device=dev)
    lp = torch.empty((R, B, Hq, Sq), dtype=torch.float32, device=dev)
    out = torch.empty((B, Hq, Sq, d), dtype=torch.float32, device=dev)
    lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=dev)
    for _ in range(3):
        m.mercury_attn_partial(qd, kd, vd, R, w["shift"], w["causal"], op, lp, stream)
        m.mercury_lse_merge(op, lp, out, lse, stream)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    t_part, t_merge = [], []
    for _ in range(reps):
        ev[0].record(stream)
        m.mercury_attn_partial(qd, kd, vd, R, w["shift"], w["causal"], op, lp, stream)
        ev[1].record(stream)
        m.mercury_lse_merge(op, lp, out, lse, stream)
        ev[2].record(stream)
        torch.cuda.synchronize(dev)
        t_part.append(ev[0].elapsed_time(ev[1]) / 1e3)
        t_merge.append(ev[1].elapsed_time(ev[2]) / 1e3)
    # the same chunk through mercury_attn_sharded: its schedule chooser cuts
    # each rank's step sequence into runs and merges them (split-KV)
    t_sh = []
    for i in range(reps + 3):
        ev[0].record(stream)
        m.mercury_attn_sharded(qd, kd, vd, R, w["shift"], w["causal"], out, lse, stream)
        ev[1].record(stream)
        torch.cuda.synchronize(dev)
        if i >= 3:
            t_sh.append(ev[0].elapsed_time(ev[1]) / 1e3)
    m.mercury_sync_status(stream)
    rows = B * Hq * Sq
    merge_bytes = R * rows * (4 * d + 4) + rows * (4 * d + 4)
    tp, tm = statistics.median(t_part), statistics.median(t_merge)
    flops = attention_flops(w)
    gbs = merge_bytes / tm / 1e9
    return {"workload": MERGE_WORKLOAD, "mode": "partial+merge",
            "partial_ms": round(tp * 1e3, 4), "attention_tflops": round(flops / tp / 1e12, 2),
            "attention_frac": round(flops / tp / 1e12 / peaks["bf16_tflops"], 4),
            "merge_ms": round(tm * 1e3, 4), "merge_bytes": merge_bytes, "merge_gbs": round(gbs, 1),
            "merge_frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4),
            "total_tflops": round(flops / (tp + tm) / 1e12, 2),
            "sharded_auto_ms": round(statistics.median(t_sh) * 1e3, 4),
            "sharded_auto_tflops": round(flops / statistics.median(t_sh) / 1e12, 2),
            "peak_kind": peak_kind, "reps": reps}


def measure_gemm(m, dev, stream, peaks, peak_kind, reps: int = 10):
    """The shifted-shard GEMM (all-gather GEMM pattern) on its workload: TFLOP/s
    of mercury_gemm_shifted (2*M*N*K flop per call)."""
    import torch

    from long_context_sharded_gb300.workloads import GEMM_WORKLOADS
    name = "gemm_m16k_k8k_n28k_r8"
    w = GEMM_WORKLOADS[name]
    g = torch.Generator().manual_seed(w["seed"])
    a = (torch.randn((w["M"], w["K"]), generator=g) * 0.5).to(torch.bfloat16).to(dev)
    b = (torch.randn((w["K"], w["N"]), generator=g) * 0.5).to(torch.bfloat16).to(dev)
    c = torch.empty((w["M"], w["N"]), dtype=torch.float32, device=dev)
    for _ in range(3):
        m.mercury_gemm_shifted(a, b, w["R"], w["shift"], c, stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        m.mercury_gemm_shifted(a, b, w["R"], w["shift"], c, stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    m.mercury_sync_status(stream)
    t = e0.elapsed_time(e1) / reps / 1e3
    flops = 2.0 * w["M"] * w["N"] * w["K"]
    return {"workload": name, "ms": round(t * 1e3, 4), "tflops": round(flops / t / 1e12, 2),
            "frac": round(flops / t / 1e12 / peaks["bf16_tflops"], 4), "peak_kind": peak_kind, "reps": reps}


def measure_decode(m, dev, stream, peaks, peak_kind, reps: int = 10):
    """One decode step of a Llama-3-70B-like model at a 128K context, batch 8
    (64 query / 8 KV heads, d 128, one query per sequence): HBM-bound, so the
    figure is GB/s of K, V, Q read and O, LSE written.  Inputs are seeded
    N(0,1) bf16 drawn on the device (4.3 GB of K/V)."""
    import torch
    B, Hq, Hkv, Sq, Skv, d = 8, 64, 8, 1, 131072, 128
    g = torch.Generator(device=dev).manual_seed(8)
    q = torch.randn((B, Hq, Sq, d), generator=g, device=dev).to(torch.bfloat16)
    k = torch.randn((B, Hkv, Skv, d), generator=g, device=dev).to(torch.bfloat16)
    v = torch.randn((B, Hkv, Skv, d), generator=g, device=dev).to(torch.bfloat16)
    out = torch.empty((B, Hq, Sq, d), dtype=torch.float32, device=dev)
    lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=dev)
    for _ in range(3):
        m.mercury_attn_decode(q, k, v, 0, False, out, lse, stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        m.mercury_attn_decode(q, k, v, 0, False, out, lse, stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    m.mercury_sync_status(stream)
    t = e0.elapsed_time(e1) / reps / 1e3
    nbytes = (q.numel() + k.numel() + v.numel()) * 2 + out.numel() * 4 + lse.numel() * 4
    return {"workload": "decode_b8_hq64_hkv8_d128_skv128k", "ms": round(t * 1e3, 4),
            "gbs": round(nbytes / t / 1e9, 1), "frac_of_hbm": round(nbytes / t / 1e9 / peaks["hbm_gbs"], 4),
            "bytes": nbytes, "peak_kind": peak_kind, "reps": reps}


# --------------------------------------------------------- reference arm

def run_reference(args):
    """The base contract's reference arm is the fp64 CPU oracle, as it stands."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from long_context_sharded_gb300.inputs import make_qkv
    w = dict(WORKLOADS[args.workload], name=args.workload)
    q, k, v = make_qkv(w["B"], w["Hq"], w["Hkv"], w["Sq"], w["Skv"], w["d"], seed=w["seed"],
                       scale=w["scale"])
    budget = max(0.5, min(3.0, 150.0 / max(1, args.steps + args.warmup)))
    for i in range(args.warmup):
        oracle_rate(q, k, v, w, seconds=budget / 4, seed=1000 + i)
    rates, times, sample = [], [], ""
    for i in range(args.steps):
        r, n, dt, sample = oracle_rate(q, k, v, w, seconds=budget, seed=w["seed"] + i)
        rates.append(r)
        times.append(dt)
    value = statistics.mean(rates)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(statistics.mean(times) * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1)*%g, bf16)" % w["scale"],
        "config": {"workload": args.workload, "B": w["B"], "Hq": w["Hq"], "Hkv": w["Hkv"], "Sq": w["Sq"],
                   "Skv": w["Skv"], "d": w["d"], "R": w["R"], "shift": w["shift"],
                   "causal": bool(w["causal"]), "mode": "oracle rows"},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": "each step: " + sample},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default=BENCH_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-e2e", action="store_true", help="do not run the host-buffer leg")
    ap.add_argument("--no-secondary", action="store_true", help="do not run the partial+merge figure")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="do not time the CPU oracle")
    ap.add_argument("--no-clocks", action="store_true", help="do not sample nvidia-smi")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.steps < 1:
        ap.error("--steps must be >= 1")
    world, _, _ = dist_env()
    if world != args.gpus:
        if args.gpus > 1 and world == 1:
            ap.error("--gpus %d needs torchrun with %d processes" % (args.gpus, args.gpus))
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
