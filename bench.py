#!/usr/bin/env python
"""Throughput benchmark of the shifted-schedule sharded attention on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...      # the fp64 CPU oracle, timed

One step = one pass of the hot path over one batch of synthetic input: a
mercury_attn_sharded call on the largest single-GPU workload, the
Llama-3-70B-like GQA prefill (B 1, 64 query / 8 KV heads, d 128, 128K tokens,
causal, R = 8 virtual ranks in the nested 2 x 4 shift order): it shards Q and
K/V, walks the shards in the shifted order, skips causally masked shards, runs
the tcgen05 attention patch and finalises O and LSE (the per-step partials are
combined on the fly, i.e. the log-sum-exp merge is fused).

The line's "configs" object times every workload on its own (CUDA events,
median of a short burst): the small MHA case, the 32K GQA causal prefill, the
batch-16 4K MHA, the headline itself, and the 2M-token MQA chunk through the
per-step partials and the separate merge, where the merge's HBM bandwidth is
reported.

Metric: attention TFLOP/s = 4 * d * (unmasked query/key pairs) * B * Hq per
step / time.  Inputs (2.5 GiB on the headline) are larger than L2, so no flush
is needed between steps.

Several GPUs (torchrun): by default virtual rank i lives on GPU i -- query
block i and KV shard i stay there and the KV shards travel between GPUs in the
shifted order (NCCL point to point, transport.py), the workload split over
the GPUs ("strong" scaling, value = the workload's FLOPs / the slowest rank's
time).  --dist-mode replicas runs independent copies of the one-GPU step
instead ("weak" scaling: all ranks' work / the slowest rank's time).
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
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM traffic of one attention launch per workload, from an ncu capture,
# valid only for the kernel source it was taken on (sha256 of the attention
# kernel's sources, first 16 hex digits).  Reported as null once the kernel
# has changed or when no capture of that workload exists.
ATTN_TRAFFIC = {
    "gqa_b1_hq32_hkv8_d128_s32k_causal_r8": {"source_sha": "50aaebb7f3354221", "bytes_per_launch": 896964864},
    "gqa_b1_hq64_hkv8_d128_s128k_causal_r8_nested2x4": {"source_sha": "50aaebb7f3354221",
                                                         "bytes_per_launch": 10273945856},
}


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


def attn_traffic(workload: str):
    """Recorded DRAM bytes of one attention launch on `workload`, or None."""
    rec = ATTN_TRAFFIC.get(workload)
    if rec and rec["source_sha"] == source_sha(*ATTN_SOURCES):
        return rec["bytes_per_launch"]
    return None


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

# Dense bf16 tensor-core work of one SM per clock: an M = 128, N = 128, K = 16
# kind::f16 MMA (524,288 FLOP) takes 64 cycles on a GB300 SM when issued back
# to back.  Times the SM count and the sampled SM clock, this is the tensor
# pipe's ceiling at the clock the kernel actually ran at.
TENSOR_FLOP_PER_CYCLE_PER_SM = 8192


def device_qkv(w, dev):
    from long_context_sharded_gb300.inputs import make_qkv
    q, k, v = make_qkv(w["B"], w["Hq"], w["Hkv"], w["Sq"], w["Skv"], w["d"], seed=w["seed"], scale=w["scale"])
    return q, k, v, q.to(dev), k.to(dev), v.to(dev)


def launches_per_call(m, w, n_sms: int) -> int:
    """Kernels one mercury_attn_sharded call launches: 1 for the fused
    schedule, 2 when the library's chooser splits it (attention + merge),
    as the library itself reports its choice for this shape."""
    runs = m.mercury_choose_runs(w["B"], w["Hq"], w["Hkv"], w["Sq"], w["Skv"], w["d"], w["causal"],
                                 w["R"], w["shift"], n_sms)
    return 1 if runs == 1 else 2


def clock_peak_tflops(n_sms: int, sm_mhz):
    if not sm_mhz:
        return None
    return TENSOR_FLOP_PER_CYCLE_PER_SM * n_sms * sm_mhz * 1e6 / 1e12


def time_calls(fn, stream, reps: int, warmup: int = 3):
    """CUDA-event time of each of `reps` calls of fn on `stream` (ms)."""
    import torch
    for _ in range(warmup):
        fn()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    torch.cuda.synchronize()
    ev[0].record(stream)
    for i in range(reps):
        fn()
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    return [ev[i].elapsed_time(ev[i + 1]) for i in range(reps)]


def measure_config(m, name, dev, stream, peaks, n_sms, reps):
    """One workload, timed on its own: the fused call (mercury_attn_sharded),
    or for the partial-mode workload the per-step partials and the merge
    separately plus the same chunk through mercury_attn_sharded's own
    schedule.  Each figure is the median of `reps` back-to-back calls (CUDA
    events on the launching stream); a short burst, so fractions are of the
    burst peak."""
    import torch
    w = dict(WORKLOADS[name], name=name)
    B, Hq, Sq, d, R = w["B"], w["Hq"], w["Sq"], w["d"], w["R"]
    _, _, _, qd, kd, vd = device_qkv(w, dev)
    flops = attention_flops(w)
    out = torch.empty((B, Hq, Sq, d), dtype=torch.float32, device=dev)
    lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=dev)
    burst = peaks["bf16_tflops"]
    res = {"mode": "fused" if w["mode"] == "fused" else "partial+merge", "reps": reps, "flop": flops}
    if w["mode"] == "fused":
        tw0 = time.time()
        ms = statistics.median(time_calls(
            lambda: m.mercury_attn_sharded(qd, kd, vd, R, w["shift"], w["causal"], out, lse, stream), stream, reps))
        res["window"] = (tw0, time.time())
        tf = flops / (ms / 1e3) / 1e12
        res.update({"ms": round(ms, 4), "tflops": round(tf, 2), "frac": round(tf / burst, 4),
                    "launches_per_call": launches_per_call(m, w, n_sms)})
    else:
        op = torch.empty((R, B, Hq, Sq, d), dtype=torch.float32, device=dev)
        lp = torch.empty((R, B, Hq, Sq), dtype=torch.float32, device=dev)
        tw0 = time.time()
        tp = statistics.median(time_calls(
            lambda: m.mercury_attn_partial(qd, kd, vd, R, w["shift"], w["causal"], op, lp, stream), stream, reps))
        res["window"] = (tw0, time.time())
        tm = statistics.median(time_calls(lambda: m.mercury_lse_merge(op, lp, out, lse, stream), stream, reps))
        ts = statistics.median(time_calls(
            lambda: m.mercury_attn_sharded(qd, kd, vd, R, w["shift"], w["causal"], out, lse, stream), stream, reps))
        rows = B * Hq * Sq
        merge_bytes = (R + 1) * rows * (4 * d + 4)
        gbs = merge_bytes / (tm / 1e3) / 1e9
        res.update({"partial_ms": round(tp, 4), "attention_tflops": round(flops / (tp / 1e3) / 1e12, 2),
                    "attention_frac": round(flops / (tp / 1e3) / 1e12 / burst, 4),
                    "merge_ms": round(tm, 4), "merge_bytes": merge_bytes, "merge_gbs": round(gbs, 1),
                    "merge_frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4),
                    "ms": round(tp + tm, 4), "tflops": round(flops / ((tp + tm) / 1e3) / 1e12, 2),
                    "frac": round(flops / ((tp + tm) / 1e3) / 1e12 / burst, 4),
                    "sharded_auto_ms": round(ts, 4),
                    "sharded_auto_tflops": round(flops / (ts / 1e3) / 1e12, 2)})
        del op, lp
    m.mercury_sync_status(stream)
    del qd, kd, vd, out, lse
    torch.cuda.empty_cache()
    return res


def attach_config_clocks(configs, rows, n_sms):
    """Each timed workload's own median SM clock (nvidia-smi samples inside
    its timed calls, warm-up included) and its TFLOP/s as a fraction of the
    tensor pipe's ceiling at that clock: a burst long enough to reach the
    power cap shows as a lower clock, not a lower fraction.  Bursts shorter
    than the 25 ms sampling interval may carry no sample (null)."""
    for name, cfg in configs.items():
        if not isinstance(cfg, dict) or "window" not in cfg:
            continue
        t0, t1 = cfg.pop("window")
        s = ClockSampler.summarise(rows, t0, t1) if rows else {"sm_mhz": None, "samples": 0}
        mhz = s["sm_mhz"]
        tf = cfg.get("attention_tflops", cfg.get("tflops"))
        cp = clock_peak_tflops(n_sms, mhz)
        cfg["sm_mhz"] = mhz
        cfg["clock_samples"] = s["samples"]
        cfg["clock_frac"] = round(tf / cp, 4) if cp and tf else None


def run_gpu(args):
    import torch

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    from long_context_sharded_gb300 import mercury as m

    w = dict(WORKLOADS[args.workload], name=args.workload)
    B, Hq, Hkv, Sq, Skv, d = w["B"], w["Hq"], w["Hkv"], w["Sq"], w["Skv"], w["d"]
    R, shift, causal = w["R"], w["shift"], w["causal"]
    partial = w["mode"] == "partial"
    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    flops = attention_flops(w)
    q, k, v, qd, kd, vd = device_qkv(w, dev)
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

    launches_per_step = 2 if partial else launches_per_call(m, w, n_sms)
    for _ in range(args.warmup):
        step()
    m.mercury_sync_status(stream)

    sampler = ClockSampler(local)
    sampling = rank == 0 and not args.no_clocks
    if sampling:
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
    m.mercury_sync_status(stream)
    per_step_ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    elapsed_s = ev[0].elapsed_time(ev[args.steps]) / 1e3
    max_s = max_over_ranks(elapsed_s, world, dev)
    value = aggregate_value(flops, args.steps, world, max_s) / 1e12

    # End to end through the public API with host buffers: every step copies
    # its inputs from pinned host memory to the device, runs the call and
    # copies O and LSE back.  Steps are pipelined the way a caller streaming
    # batches would: two device buffer slots, H2D on one stream, compute on
    # another, D2H on a third, so step i's copies overlap step i-1's compute.
    # The copies' own durations (CUDA events on the copy streams) give the
    # host-link rates the pipeline saw.
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
        e_steps = max(3, min(args.steps, 20))
        copy_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(e_steps + 2)]

        def e2e_step(i):
            dq_, dk_, dv_, do_, dl_, oh, lh = slots[i % 2]
            ce = copy_ev[i]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_cmp[i % 2])      # slot's inputs no longer read
                ce[0].record(s_in)
                dq_.copy_(qh, non_blocking=True)
                dk_.copy_(kh, non_blocking=True)
                dv_.copy_(vh, non_blocking=True)
                ce[1].record(s_in)
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
                ce[2].record(s_out)
                oh.copy_(do_, non_blocking=True)
                lh.copy_(dl_, non_blocking=True)
                ce[3].record(s_out)
                ev_out[i % 2].record(s_out)

        for i in range(2):
            e2e_step(e_steps + i)
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
        h2d_ms = statistics.mean(copy_ev[i][0].elapsed_time(copy_ev[i][1]) for i in range(e_steps))
        d2h_ms = statistics.mean(copy_ev[i][2].elapsed_time(copy_ev[i][3]) for i in range(e_steps))
        e2e = {"value": round(aggregate_value(flops, e_steps, world, e_s) / 1e12, 3), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e_steps,
               "h2d_gbs": round(h2d / (h2d_ms / 1e3) / 1e9, 1), "d2h_gbs": round(d2h / (d2h_ms / 1e3) / 1e9, 1),
               "h2d_ms": round(h2d_ms, 3), "d2h_ms": round(d2h_ms, 3),
               "timing": "host wall clock around the steps, all streams synchronised at both ends; "
                         "copy rates from CUDA events around each step's copies",
               "pipelining": "2 buffer slots; H2D, compute and D2H on three streams"}
        del qh, kh, vh, slots

    peaks, peak_kind = load_peaks()
    t_cfg0 = time.time()
    configs = None
    if not args.no_configs and rank == 0 and world == 1:
        configs = {"peak": peaks["bf16_tflops"],
                   "peak_kind": "%s burst bf16 (cuBLAS): each figure is a short burst of calls" % peak_kind}
        for name in WORKLOADS:
            if name == args.workload:
                continue
            reps = 100 if attention_flops(WORKLOADS[name]) < 1e10 else 10
            configs[name] = measure_config(m, name, dev, stream, peaks, n_sms, reps)
    t_cfg1 = time.time()
    rows = sampler.stop() if sampling else []
    clocks = ClockSampler.summarise(rows, t_wall0, t_wall1) if rows else None
    clocks_cfg = ClockSampler.summarise(rows, t_cfg0, t_cfg1) if rows and configs else None

    launch_ms = statistics.mean(per_step_ms)
    achieved = flops / (launch_ms / 1e3) / 1e12
    # A timed region of seconds of back-to-back tensor work runs under the
    # power cap: its fraction is of the sustained peak; a short one of the
    # burst peak.  Either way the clock-normalised fraction (achieved over the
    # tensor pipe's ceiling at the sampled median SM clock) is given too.
    long_region = elapsed_s > 1.0
    peak = peaks["bf16_tflops_sustained"] if long_region else peaks["bf16_tflops"]
    cp = clock_peak_tflops(n_sms, clocks["sm_mhz"] if clocks else None)
    roofline = {"kernel": "attn_fwd_kernel" + (" + lse_merge_kernel" if launches_per_step > 1 else ""),
                "bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "traffic": attn_traffic(args.workload),
                "peak_kind": "%s %s bf16 (cuBLAS); timed region %.2f s of back-to-back launches" % (
                    peak_kind, "sustained" if long_region else "burst", elapsed_s),
                "frac_of_burst": round(achieved / peaks["bf16_tflops"], 4),
                "frac_of_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4),
                "clock_peak": None if cp is None else {
                    "tflops": round(cp, 1), "sm_mhz": clocks["sm_mhz"], "frac": round(achieved / cp, 4),
                    "basis": "%d FLOP/cycle/SM x %d SMs x median SM clock in the timed region" % (
                        TENSOR_FLOP_PER_CYCLE_PER_SM, n_sms)},
                "algorithmic_flop_per_launch": flops,
                "algorithmic_bytes_per_launch": (q.numel() + k.numel() + v.numel()) * 2
                + out.numel() * 4 + lse.numel() * 4}
    if configs is not None:
        headline = {"mode": "fused" if not partial else "partial+merge", "ms": round(statistics.median(per_step_ms), 4),
                    "tflops": round(achieved, 2), "frac": round(achieved / peaks["bf16_tflops"], 4),
                    "flop": flops, "source": "the headline timed region (%d steps)" % args.steps,
                    "launches_per_call": launches_per_step,
                    "sm_mhz": clocks["sm_mhz"] if clocks else None,
                    "clock_frac": round(achieved / cp, 4) if cp else None}
        configs = dict([(k_, v_) for k_, v_ in configs.items() if k_ in ("peak", "peak_kind")]
                       + [(n, headline if n == args.workload else configs[n]) for n in WORKLOADS])
        configs["clocks"] = clocks_cfg
        attach_config_clocks(configs, rows, n_sms)
        torch.cuda.empty_cache()
        # the schedule planner's estimate (built-in profile) beside the measured time
        prof = m.mercury_default_cost_profile(n_sms)
        top = m.mercury_plan_schedules(B, Hq, Hkv, Sq, Skv, d, causal, R, shift, 0, prof, 1)[0][0]
        configs["schedule_model"] = {"workload": args.workload, "schedule": [top.R, top.Rq, top.n_runs],
                                     "schedule_keys": ["R", "Rq", "n_runs"],
                                     "predicted_ms": round(top.predicted_us / 1e3, 4),
                                     "measured_ms": round(statistics.median(per_step_ms), 4)}

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
            "configs": configs, "gemm": gemm, "decode": decode,
            "per_step_ms": {"min": round(min(per_step_ms), 4), "median": round(statistics.median(per_step_ms), 4),
                            "max": round(max(per_step_ms), 4)},
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ------------------------------------------------- N GPUs: the shifted exchange

def dist_shift_for(world: int, shift: int) -> int:
    """Shift order across `world` devices: the workload's nested inner size
    when it divides the device count into two or more groups, else flat."""
    if shift >= 2 and world % shift == 0 and world > shift:
        return shift
    return 1


def local_block(t, rank: int, world: int):
    """Rank `rank`'s contiguous block of the sequence axis (dim 2) of t."""
    n = t.shape[2] // world
    return t[:, :, rank * n:(rank + 1) * n].contiguous()


def run_gpu_shifted(args):
    """Virtual rank i on GPU i: query block i and KV shard i stay on GPU i,
    the shards travel between GPUs in the shifted order (NCCL point to point
    into a local double buffer, see transport.py) and every GPU runs the
    local patch and the merge on its own memory.  The whole workload is split
    over the GPUs, so the scaling is strong; value = the workload's FLOPs per
    step / the slowest rank's time."""
    import torch

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    os.environ.setdefault("NCCL_NVLS_ENABLE", "0")
    dist = init_dist(world, "nccl")
    from long_context_sharded_gb300 import mercury as m  # noqa: F401  (loads the library)
    from long_context_sharded_gb300 import transport as tp
    from long_context_sharded_gb300.inputs import make_qkv

    w = dict(WORKLOADS[args.workload], name=args.workload)
    B, Hq, Hkv, Sq, Skv, d, causal = w["B"], w["Hq"], w["Hkv"], w["Sq"], w["Skv"], w["d"], w["causal"]
    if Sq % world or Skv % world or (causal and Sq != Skv):
        raise SystemExit("workload %s cannot be split over %d GPUs" % (args.workload, world))
    shift = dist_shift_for(world, w["shift"])
    flops = attention_flops(w)
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, d, seed=w["seed"], scale=w["scale"])
    qh, kh, vh = (local_block(t, rank, world) for t in (q, k, v))
    del q, k, v
    qb, kb, vb = qh.to(dev), kh.to(dev), vh.to(dev)
    ex = tp.ShiftedKV(world, shift, causal, rank)
    order = tp.shift_table(world, shift)
    n_patch = sum(1 for s in order[rank] if not causal or tp.causal_relation(rank, int(s)) != "none")

    def step():
        return ex.run(qb, kb, vb, tp.cuda_patch, tp.cuda_merge)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # rank 0 samples its own GPU's clocks during the timed region
    sampler = ClockSampler(local)
    sampling = rank == 0 and not args.no_clocks
    if sampling:
        sampler.start()
    barrier(world)
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    ev0.record(stream)
    for _ in range(args.steps):
        o, l = step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    barrier(world)
    rows = sampler.stop() if sampling else []
    clocks = ClockSampler.summarise(rows, t_wall0, t_wall1) if rows else None
    max_s = max_over_ranks(ev0.elapsed_time(ev1) / 1e3, world, dev)
    value = flops * args.steps / max_s / 1e12

    # end to end: this rank's blocks from pinned host memory, its O and LSE back
    qp, kp, vp = qh.pin_memory(), kh.pin_memory(), vh.pin_memory()
    oh = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    lh = torch.empty(l.shape, dtype=l.dtype, pin_memory=True)
    e_steps = max(3, min(args.steps, 10))
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(e_steps):
        qb.copy_(qp, non_blocking=True)
        kb.copy_(kp, non_blocking=True)
        vb.copy_(vp, non_blocking=True)
        o, l = step()
        oh.copy_(o, non_blocking=True)
        lh.copy_(l, non_blocking=True)
    torch.cuda.synchronize(dev)
    e_s = max_over_ranks(time.perf_counter() - t0, world, dev)
    m.mercury_sync_status(stream)
    if rank == 0:
        h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh)) * world
        d2h = (o.numel() * o.element_size() + l.numel() * l.element_size()) * world
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(max_s * 1e3 / args.steps, 4), "higher_is_better": True,
            "scaling": "strong", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1)*%g, bf16)" % w["scale"],
            "config": {"workload": args.workload, "B": B, "Hq": Hq, "Hkv": Hkv, "Sq": Sq, "Skv": Skv, "d": d,
                       "R": world, "shift": shift, "causal": bool(causal), "mode": "fused per step + merge",
                       "parallelism": "shifted KV exchange over %d GPUs (NCCL point to point)" % world,
                       "l2": "inputs larger than L2, no flush"},
            "gpu_launches": args.steps * (n_patch + max(0, n_patch - 1)),
            "e2e": {"value": round(flops * e_steps / e_s / 1e12, 3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e_steps},
            "roofline": None, "cpu_baseline": None, "clocks": clocks,
            "note": "rank 0's line (clocks: rank 0's GPU); the per-rank causal work is uneven (rank i runs i + 1 of the %d shards)"
                    % world if causal else "rank 0's line",
        }
        print(json.dumps(line), flush=True)
    dist.destroy_process_group()


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
    ap.add_argument("--no-configs", action="store_true", help="do not time the other workloads")
    ap.add_argument("--no-secondary", action="store_true", help="do not time the GEMM and decode figures")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="do not time the CPU oracle")
    ap.add_argument("--no-clocks", action="store_true", help="do not sample nvidia-smi")
    ap.add_argument("--dist-mode", choices=["shifted", "replicas"], default="shifted",
                    help="with several GPUs: split the workload over them and exchange KV shards in the "
                         "shifted order (default), or run independent replicas")
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
    elif world > 1 and args.dist_mode == "shifted":
        run_gpu_shifted(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
