"""mercury_attn_split_noalloc: split-KV attention for callers that cannot
allocate device memory (an allocator or memory manager calling attention from
inside itself, serving loops that forbid allocator calls on the hot path,
hosts with a fixed device-memory budget).  Its partials live in a fixed
64 MiB array of the library's module instead of allocated scratch.

Called through the C ABI with raw device pointers, on two calls in a row (the
shared array keeps the first call's contents when the second one runs), and
checked with the parity tolerances of the other GPU tests against both
mercury_attn_sharded (the allocating entry point) and the fp64 CPU oracle.
Around the second call neither the device's free memory nor torch's
allocation count may change: the call must not allocate.  This file sorts
last so a run that stops at the first failure has run every other test
already; it also passes alone in a fresh process (the first call does the
per-device set-up, which loads the array's module).
"""
import ctypes
import gc

import numpy as np
import pytest
import torch

import oracle
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


def check_close(o, l, o_ref, l_ref, what):
    o = np.asarray(o, dtype=np.float64)
    l = np.asarray(l, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    l_ref = np.asarray(l_ref, dtype=np.float64)
    assert np.isfinite(o).all(), what
    err = np.abs(o - o_ref)
    assert err.max() <= O_MAX and err.mean() <= O_MEAN, (what, err.max(), err.mean())
    fin = np.isfinite(l_ref)
    assert (np.isfinite(l) == fin).all(), what
    assert np.abs(l[fin] - l_ref[fin]).max() <= LSE_MAX, what


@pytest.mark.parametrize("cfg", [
    # B, Hq, Hkv, Sq, Skv, d, R, shift, causal, n_runs
    (1, 8, 1, 512, 32768, 128, 16, 1, False, 4),
    (1, 4, 2, 1024, 2048, 64, 8, 4, True, 3),
], ids=["mqa_long_kv", "gqa_causal_nested"])
def test_noalloc_matches_sharded_and_oracle_two_calls(m, cfg):
    B, Hq, Hkv, Sq, Skv, d, R, shift, causal, n_runs = cfg
    for call, seed in enumerate((11, 12)):
        q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, d, seed=seed + sum(cfg[:7]))
        qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
        out = torch.empty((B, Hq, Sq, d), dtype=torch.float32, device="cuda")
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device="cuda")
        # the allocating entry point's result, taken before the bracket
        o_sh, l_sh = m.mercury_attn_sharded(qd, kd, vd, R, shift, causal)
        m.mercury_sync_status()
        # no garbage collection inside the bracket: a collected cycle holding a
        # CUDA tensor would change torch's count without any allocation here
        gc.collect()
        gc.disable()
        try:
            free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
            rc = noalloc_call(m, qd, kd, vd, R, shift, causal, n_runs, out, lse)
            assert rc == 0, m.lib.mercury_last_error()
            m.mercury_sync_status()
            free1, alloc1 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
        finally:
            gc.enable()
        if call == 1:
            # the first call on a device may load the array's module; later
            # calls allocate nothing
            assert free1 == free0 and alloc1 == alloc0, (free0, free1, alloc0, alloc1)
        check_close(out.cpu().numpy(), lse.cpu().numpy(), o_sh.cpu().numpy(), l_sh.cpu().numpy(),
                    "vs mercury_attn_sharded, call %d" % call)
        o_ref, l_ref = oracle.attn(q, k, v, causal)
        check_close(out.cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, "vs oracle, call %d" % call)


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


def test_noalloc_follows_the_wait_budget_and_fault_hook(m, monkeypatch):
    """Like every other call, the allocation-free call takes its wait budget
    from MERCURY_WAIT_NS and the test fault hook from MERCURY_FAULT: a dropped
    arrive makes a wait run out after 20 ms, the status reports it, and the
    next call is correct."""
    B, Hq, Hkv, Sq, Skv, d, R, n_runs = 1, 4, 1, 256, 4096, 128, 8, 2
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, d, seed=5)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out = torch.empty((B, Hq, Sq, d), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device="cuda")
    monkeypatch.setenv("MERCURY_FAULT", "drop_p_arrive")
    monkeypatch.setenv("MERCURY_WAIT_NS", "20000000")
    assert noalloc_call(m, qd, kd, vd, R, 1, False, n_runs, out, lse) == 0
    with pytest.raises(m.MercuryError) as e:
        m.mercury_sync_status()
    assert e.value.status == m.MERCURY_ETIMEOUT
    monkeypatch.delenv("MERCURY_FAULT")
    monkeypatch.delenv("MERCURY_WAIT_NS")
    assert noalloc_call(m, qd, kd, vd, R, 1, False, n_runs, out, lse) == 0
    m.mercury_sync_status()
    o_ref, l_ref = oracle.attn(q, k, v, False)
    check_close(out.cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, "after the timeout")
