"""mercury_attn_split_noalloc: split-KV attention for callers that cannot
allocate device memory (an allocator or memory manager calling attention from
inside itself, serving loops that forbid allocator calls on the hot path,
hosts with a fixed device-memory budget).  Its partials live in a fixed
64 MiB array of the library's module instead of allocated scratch.

Called through the C ABI with raw device pointers and checked against
mercury_attn_sharded, the allocating entry point, with the parity tolerances
of the other GPU tests, on two calls in a row (the shared array keeps the
first call's contents when the second one runs).  This file sorts last so a
run that stops at the first failure has run every other test already; it also
passes alone in a fresh process (the first call does the per-device set-up).
"""
import ctypes

import numpy as np
import pytest
import torch

from long_context_sharded_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3


@pytest.fixture(scope="module")
def m():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_sharded_gb300 import build
    build.build()
    from long_context_sharded_gb300 import mercury
    return mercury


def noalloc_call(m, q, k, v, R, shift, causal, n_runs, out, lse):
    """One call of the C entry point with raw pointers on the current stream."""
    B, Hq, Sq, d = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    stream = torch.cuda.current_stream().cuda_stream
    return m.lib.mercury_attn_split_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
        B, Hq, Hkv, Sq, Skv, d, R, shift, int(causal), n_runs,
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()), ctypes.c_void_p(stream))


def check_against_sharded(m, o_na, l_na, o_ref, l_ref):
    torch.cuda.synchronize()
    diff = (o_na - o_ref).abs()
    assert torch.isfinite(o_na).all()
    assert diff.max().item() <= O_MAX and diff.mean().item() <= O_MEAN, (diff.max().item(),
                                                                         diff.mean().item())
    fin = torch.isfinite(l_ref)
    assert torch.equal(torch.isfinite(l_na), fin)
    assert (l_na[fin] - l_ref[fin]).abs().max().item() <= LSE_MAX


@pytest.mark.parametrize("cfg", [
    # B, Hq, Hkv, Sq, Skv, d, R, shift, causal, n_runs
    (1, 8, 1, 512, 32768, 128, 16, 1, False, 4),
    (1, 4, 2, 1024, 2048, 64, 8, 4, True, 3),
], ids=["mqa_long_kv", "gqa_causal_nested"])
def test_noalloc_matches_sharded_two_calls(m, cfg):
    B, Hq, Hkv, Sq, Skv, d, R, shift, causal, n_runs = cfg
    for call, seed in enumerate((11, 12)):
        q, k, v = (x.cuda() for x in make_qkv(B, Hq, Hkv, Sq, Skv, d, seed=seed + sum(cfg[:7])))
        out = torch.empty((B, Hq, Sq, d), dtype=torch.float32, device="cuda")
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device="cuda")
        rc = noalloc_call(m, q, k, v, R, shift, causal, n_runs, out, lse)
        assert rc == 0, m.lib.mercury_last_error()
        o_ref, l_ref = m.mercury_attn_sharded(q, k, v, R, shift, causal)
        m.mercury_sync_status()
        check_against_sharded(m, out, lse, o_ref, l_ref)


def test_noalloc_rejects_oversized_partials(m):
    # 64 runs x 8*2048 rows x 129 x 4 bytes = 541 MB > the 64 MiB array
    B, Hq, Hkv, Sq, Skv, d, R = 1, 8, 1, 2048, 8192, 128, 64
    q = torch.empty((B, Hq, Sq, d), dtype=torch.bfloat16, device="cuda")
    k = torch.empty((B, Hkv, Skv, d), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((B, Hq, Sq, d), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device="cuda")
    rc = noalloc_call(m, q, k, k, R, 1, False, R, out, lse)
    assert rc == m.MERCURY_EINVAL
    assert b"scratch" in m.lib.mercury_last_error()
