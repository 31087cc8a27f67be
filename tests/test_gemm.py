"""Shifted-shard GEMM: argument validation (CPU) and GPU parity against the
fp64 oracle.  Tolerance: fp32 accumulation of bf16 products over K terms,
|err| <= 1e-5 * sqrt(K) * max|a| * max|b| * 4 plus a relative 1e-5."""
import math

import numpy as np
import pytest
import torch

from oracle import gemm as og

P = 0x100000


@pytest.fixture(scope="module")
def lib():
    from long_context_sharded_gb300 import build
    build.build()
    from long_context_sharded_gb300 import mercury
    return mercury


@pytest.mark.parametrize("args,code", [
    ((0, P, 256, 256, 64, 4, 1, P), -1), ((P, P, 256, 256, 64, 4, 1, 0), -1),
    ((P, P, 250, 256, 64, 4, 1, P), -1), ((P, P, 256, 250, 64, 4, 1, P), -1),
    ((P, P, 256, 256, 60, 4, 1, P), -1), ((P, P, 256, 100, 64, 4, 1, P), -1),
    ((P, P, 256, 256, 64, 4, 3, P), -1), ((P, P, 256, 256, 64, 0, 1, P), -1),
    ((P + 2, P, 256, 256, 64, 4, 1, P), -2), ((P, P, 256, 256, 64, 4, 1, P + 4), -2),
])
def test_gemm_argument_validation(lib, args, code):
    assert lib.lib.mercury_gemm_shifted(*args, None) == code


def _rnd(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


def _check(c_gpu, a, b, rows=None):
    """c_gpu: the GPU result, or its selected rows when rows is given."""
    ref = og.gemm(a, b) if rows is None else og.gemm(a[rows], b)
    got = c_gpu
    K = a.shape[1]
    amax = a.abs().max().item() * b.abs().max().item()
    tol = 4e-5 * math.sqrt(K) * amax + 1e-5 * np.abs(ref)
    err = np.abs(got - ref)
    assert (err <= tol).all(), "max err %.3g (tol %.3g)" % (err.max(), tol.max())


@pytest.mark.gpu
@pytest.mark.parametrize("M,N,K,R,shift", [
    (128, 256, 64, 1, 1),          # one tile
    (512, 1024, 256, 4, 1),        # aligned tiles, flat shift
    (1024, 2048, 192, 8, 4),       # nested 2x4 shift
    (384, 768, 320, 2, 0),         # unshifted, K not a multiple of 64
    (200, 336, 104, 2, 1),         # ragged rows, columns, K
    (96, 128, 8, 4, 1),            # tiny blocks (24 rows per rank, 32 columns per shard)
])
def test_gemm_matches_oracle(lib, M, N, K, R, shift):
    a, b = _rnd((M, K), M + K), _rnd((K, N), N + R)
    c = lib.mercury_gemm_shifted(a.cuda(), b.cuda(), R, shift)
    lib.mercury_sync_status()
    _check(c.cpu().numpy().astype(np.float64), a, b)


@pytest.mark.gpu
def test_gemm_shift_orders_agree(lib):
    a, b = _rnd((1024, 512), 1), _rnd((512, 2048), 2)
    ad, bd = a.cuda(), b.cuda()
    outs = [lib.mercury_gemm_shifted(ad, bd, 8, s) for s in (0, 1, 2, 4, 8)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])   # same tiles, same K order: bit-identical


@pytest.mark.gpu
def test_gemm_workload_sampled_rows(lib):
    from long_context_sharded_gb300.workloads import GEMM_WORKLOADS
    w = GEMM_WORKLOADS["gemm_m16k_k8k_n28k_r8"]
    a = _rnd((w["M"], w["K"]), w["seed"], 0.5)
    b = _rnd((w["K"], w["N"]), w["seed"] + 1, 0.5)
    c = lib.mercury_gemm_shifted(a.cuda(), b.cuda(), w["R"], w["shift"])
    lib.mercury_sync_status()
    g = torch.Generator().manual_seed(3)
    Mr = w["M"] // w["R"]
    rows = sorted(set([0, w["M"] - 1] + [i * Mr for i in range(w["R"])] + [i * Mr - 1 for i in range(1, w["R"])]
                      + torch.randint(0, w["M"], (48,), generator=g).tolist()))
    _check(c[rows].cpu().numpy().astype(np.float64), a, b, rows=rows)
