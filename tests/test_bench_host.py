"""Host logic of bench.py without a GPU: max-over-ranks timing and whole-job
throughput across two gloo ranks (the replica path of --gpus N), clock-log
parsing, per-workload clocks, and the reference arm's rank filter."""
import json
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    bench.init_dist(world, "gloo")
    elapsed = [0.5, 2.0][rank]           # rank 1 is the slow one
    mx = bench.max_over_ranks(elapsed, world)
    bench.barrier(world)
    value = bench.aggregate_value(1e12, 10, world, mx)
    q.put((rank, mx, value))
    dist.destroy_process_group()


def test_two_rank_max_timing_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, value in res:
        assert mx == 2.0                              # both ranks see the slowest time
        assert value == pytest.approx(1e12 * 10 * 2 / 2.0)


def test_single_rank_identity():
    assert bench.max_over_ranks(1.25, 1) == 1.25
    assert bench.aggregate_value(2.0, 3, 1, 1.5) == pytest.approx(4.0)


def test_clock_summary_parsing():
    rows = [
        ["2026/12/02 10:00:00.100", "0", "1965 MHz", "2070 MHz", "900.1 W", "0x0", "Not Active",
         "Not Active", "Not Active", "Not Active"],
        ["2026/12/02 10:00:00.200", "0", "1980 MHz", "2070 MHz", "1200.0 W", "0x4", "Not Active",
         "Not Active", "Not Active", "Active"],
        ["2026/12/02 10:00:09.000", "0", "500 MHz", "2070 MHz", "90.0 W", "0x0", "Active",
         "Not Active", "Not Active", "Not Active"],   # outside the window
    ]
    import datetime
    t0 = datetime.datetime(2026, 12, 2, 10, 0, 0).timestamp()
    s = bench.ClockSampler.summarise(rows, t0, t0 + 1.0)
    assert s["samples"] == 2 and s["sm_mhz"] == pytest.approx(1972.5)
    assert s["sm_max_mhz"] == 2070 and s["reasons"] == ["sw_power_cap"]


def test_reference_arm_nonzero_rank_does_nothing(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.run_reference(bench_args())
    assert capsys.readouterr().out == ""


def bench_args():
    import argparse
    return argparse.Namespace(workload="mha_b1_h4_d64_s512_r4", steps=1, warmup=3)


def test_shift_order_across_devices():
    """With several GPUs the workload's nested order keeps its inner size when
    that splits the GPUs into two or more groups; otherwise the flat order."""
    assert bench.dist_shift_for(8, 4) == 4
    assert bench.dist_shift_for(8, 2) == 2
    assert bench.dist_shift_for(4, 4) == 1
    assert bench.dist_shift_for(2, 4) == 1
    assert bench.dist_shift_for(4, 1) == 1
    assert bench.dist_shift_for(6, 4) == 1


def test_local_blocks_tile_the_sequence():
    import torch
    t = torch.arange(2 * 3 * 16 * 4).view(2, 3, 16, 4)
    parts = [bench.local_block(t, r, 4) for r in range(4)]
    assert all(p.shape == (2, 3, 4, 4) and p.is_contiguous() for p in parts)
    assert torch.equal(torch.cat(parts, dim=2), t)


def test_clock_normalised_ceiling():
    """8192 FLOP/cycle/SM x SMs x MHz: 152 SMs at 2070 MHz is 2577.5 TFLOP/s."""
    assert bench.clock_peak_tflops(152, 2070) == pytest.approx(8192 * 152 * 2070e6 / 1e12)
    assert bench.clock_peak_tflops(152, 2070) == pytest.approx(2577.5, abs=0.1)
    assert bench.clock_peak_tflops(152, None) is None


def test_config_clocks_from_each_window():
    """Every timed workload gets the median SM clock of the samples inside its
    own timed calls and its TFLOP/s over the tensor ceiling at that clock; a
    window with no sample gets null; the window itself leaves the record."""
    import datetime
    t0 = datetime.datetime(2026, 12, 2, 10, 0, 0).timestamp()
    row = lambda sec, mhz: ["2026/12/02 10:00:%06.3f" % sec, "0", "%d MHz" % mhz, "2070 MHz", "1000.0 W",
                            "0x4", "Not Active", "Not Active", "Not Active", "Active"]
    rows = [row(0.10, 2070), row(0.12, 2070), row(0.50, 1750), row(0.52, 1760), row(0.54, 1770)]
    configs = {
        "peak": 1902.6,
        "a": {"tflops": 1800.0, "window": (t0 + 0.05, t0 + 0.2)},
        "b": {"attention_tflops": 1700.0, "tflops": 1690.0, "window": (t0 + 0.45, t0 + 0.6)},
        "c": {"tflops": 10.0, "window": (t0 + 0.3, t0 + 0.31)},
        "clocks": {"sm_mhz": 2070},
    }
    bench.attach_config_clocks(configs, rows, 152)
    assert configs["a"]["sm_mhz"] == 2070 and configs["a"]["clock_samples"] == 2
    assert configs["a"]["clock_frac"] == pytest.approx(1800.0 / bench.clock_peak_tflops(152, 2070), abs=1e-4)
    assert configs["b"]["sm_mhz"] == 1760
    assert configs["b"]["clock_frac"] == pytest.approx(1700.0 / bench.clock_peak_tflops(152, 1760), abs=1e-4)
    assert configs["c"]["sm_mhz"] is None and configs["c"]["clock_frac"] is None
    assert all("window" not in v for v in configs.values() if isinstance(v, dict))
    json.dumps(configs)


def test_launches_per_call_follows_the_library_schedule(monkeypatch):
    """The bench's launch count per mercury_attn_sharded call mirrors the
    library's run-count choice: one launch for the fused workloads, attention
    plus merge when the chooser splits (the 2M-token chunk)."""
    from long_context_sharded_gb300 import build
    build.build()
    from long_context_sharded_gb300 import mercury as m
    from long_context_sharded_gb300.workloads import WORKLOADS
    monkeypatch.delenv("MERCURY_SPLIT_GROUPS", raising=False)
    assert bench.launches_per_call(m, WORKLOADS["gqa_b1_hq64_hkv8_d128_s128k_causal_r8_nested2x4"], 152) == 1
    assert bench.launches_per_call(m, WORKLOADS["gqa_b1_hq32_hkv8_d128_s32k_causal_r8"], 152) == 1
    assert bench.launches_per_call(m, WORKLOADS["mqa_b1_hq8_hkv1_d128_sq2k_skv2m_r64_merge"], 152) == 2
    monkeypatch.setenv("MERCURY_SPLIT_GROUPS", "1")
    assert bench.launches_per_call(m, WORKLOADS["mqa_b1_hq8_hkv1_d128_sq2k_skv2m_r64_merge"], 152) == 1
