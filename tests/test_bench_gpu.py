"""bench.py's multi-GPU path (the shifted KV exchange of `--gpus N` under
torchrun) run as a single rank on one GPU: one NCCL process group of size
one, so the exchange is trivial, but the timing, the end-to-end leg, the clock
record and the JSON line are the ones an N-GPU run prints."""
import argparse
import json
import socket

import pytest
import torch

import bench

pytestmark = pytest.mark.gpu


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_shifted_bench_path_on_one_rank(monkeypatch, capsys):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_sharded_gb300 import build
    build.build()
    import torch.distributed as dist
    for k, v in dict(WORLD_SIZE="1", RANK="0", LOCAL_RANK="0", MASTER_ADDR="127.0.0.1",
                     MASTER_PORT=str(_free_port())).items():
        monkeypatch.setenv(k, v)
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", rank=0, world_size=1)
    try:
        args = argparse.Namespace(gpus=1, steps=2, warmup=3, impl="native",
                                  workload="gqa_b1_hq32_hkv8_d128_s32k_causal_r8", cpu_seconds=0,
                                  no_e2e=False, no_configs=True, no_secondary=True, no_cpu_baseline=True,
                                  no_clocks=True, dist_mode="shifted")
        bench.run_gpu_shifted(args)
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["n_gpus"] == 1 and line["scaling"] == "strong" and line["steps"] == 2
    assert line["value"] > 100 and line["e2e"]["value"] > 0
    assert line["gpu_launches"] == 2 and line["config"]["R"] == 1
    assert "clocks" in line
