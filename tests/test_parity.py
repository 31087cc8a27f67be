"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle.

Tolerances (bf16 inputs, fp32 accumulation, P rounded to bf16 before P.V):
  O:   max |gpu - oracle| <= 2e-2 and mean |gpu - oracle| <= 2e-3
  LSE: max |gpu - oracle| <= 1e-3
Small shapes are compared on every row; the full-size workloads on a seeded
row sample (block edges, the diagonal, random rows), plus a full-coverage
cross-check of the fused path against partials + merge on the GPU.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from long_context_sharded_gb300.inputs import make_qkv, sample_rows
from long_context_sharded_gb300.workloads import WORKLOADS

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


def assert_close(o_gpu, l_gpu, o_ref, l_ref, what=""):
    o_gpu = np.asarray(o_gpu, dtype=np.float64).reshape(o_ref.shape)
    l_gpu = np.asarray(l_gpu, dtype=np.float64).reshape(l_ref.shape)
    assert np.isfinite(o_gpu).all(), what + ": non-finite O"
    fin = np.isfinite(l_ref)
    assert (np.isfinite(l_gpu) == fin).all(), what + ": LSE finiteness differs"
    err = np.abs(o_gpu - o_ref)
    lerr = np.abs(l_gpu[fin] - l_ref[fin]) if fin.any() else np.zeros(1)
    msg = "%s: O max %.3g mean %.3g, LSE max %.3g" % (what, err.max(), err.mean(), lerr.max())
    assert err.max() <= O_MAX, msg
    assert err.mean() <= O_MEAN, msg
    assert lerr.max() <= LSE_MAX, msg


def run_sharded(m, q, k, v, R, shift, causal):
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out, lse = m.mercury_attn_sharded(qd, kd, vd, R, shift, causal)
    m.mercury_sync_status()
    return out.cpu().numpy(), lse.cpu().numpy()


def run_partial_merge(m, q, k, v, R, shift, causal):
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    op, lp = m.mercury_attn_partial(qd, kd, vd, R, shift, causal)
    out, lse = m.mercury_lse_merge(op, lp)
    m.mercury_sync_status()
    return op.cpu().numpy(), lp.cpu().numpy(), out.cpu().numpy(), lse.cpu().numpy()


# ------------------------------------------------ structured probes (S vs PV)

@pytest.mark.parametrize("d", [64, 128])
def test_probe_q_zero_mean_of_v(m, d):
    """Q = 0: every score is 0, so O is the mean of V -- exercises P.V alone."""
    _, k, v = make_qkv(1, 1, 1, 256, 256, d, seed=101)
    q = torch.zeros(1, 1, 256, d, dtype=torch.bfloat16)
    out, lse = run_sharded(m, q, k, v, 1, 1, False)
    vv = v.to(torch.float64).numpy()[0, 0]
    np.testing.assert_allclose(out[0, 0], np.broadcast_to(vv.mean(0), (256, d)), atol=2e-3)
    np.testing.assert_allclose(lse[0, 0], math.log(256), atol=1e-4)


@pytest.mark.parametrize("d", [64, 128])
def test_probe_one_hot_selects_row(m, d):
    """Dominant one-hot scores: query i and key j share coordinate (index mod d),
    so row i attends (almost) only to keys j = i mod d -- exercises Q.K^T."""
    S = 256
    alpha = 16.0 if d == 64 else 24.0
    q = torch.zeros(1, 1, S, d)
    k = torch.zeros(1, 1, S, d)
    idx = torch.arange(S)
    q[0, 0, idx, idx % d] = alpha
    k[0, 0, idx, (idx * 3) % d] = alpha
    _, _, v = make_qkv(1, 1, 1, S, S, d, seed=5)
    q, k = q.to(torch.bfloat16), k.to(torch.bfloat16)
    out, lse = run_sharded(m, q, k, v, 1, 1, False)
    o_ref, l_ref = oracle.attn(q, k, v, False)
    assert_close(out, lse, o_ref, l_ref, "one-hot")


# ------------------------------------------------------ small shapes, all rows

SMALL = [
    # B, Hq, Hkv, Sq, Skv, d, R, shift, causal
    (1, 4, 4, 512, 512, 64, 4, 1, False),      # the small MHA workload
    (1, 1, 1, 128, 128, 128, 1, 1, False),     # one tile
    (1, 2, 1, 256, 256, 128, 2, 1, True),      # GQA pair, causal diagonal
    (2, 4, 2, 384, 384, 128, 3, 1, True),      # odd R, causal
    (1, 8, 2, 512, 512, 64, 4, 0, True),       # unshifted order
    (1, 8, 8, 1024, 1024, 128, 8, 4, True),    # nested 2x4 shift, MHA row pairs
    (1, 8, 1, 128, 4096, 128, 4, 1, False),    # MQA, heads packed 4 per tile (Bq = 32)
    (1, 8, 2, 96, 96, 64, 3, 1, True),         # Bq = 32, G = 4 packed, causal
    (1, 3, 1, 200, 200, 128, 2, 1, True),      # ragged block and shard, odd group
    (2, 2, 2, 384, 384, 64, 3, 1, False),      # MHA odd tile count
    (1, 6, 3, 64, 192, 128, 8, 2, True),       # Bq = 8, Sq < Skv causal, nested
    (1, 4, 1, 16, 16, 128, 1, 1, True),        # tiny
    (1, 2, 2, 1000, 1000, 128, 1, 1, True),    # Skv not a multiple of 128
    (1, 2, 2, 1024, 1024, 64, 128, 1, True),   # the largest R: 8-row blocks and shards
    (1, 4, 1, 512, 2048, 128, 4, 1, True),     # causal, Sq < Skv (bottom-right alignment)
    (3, 4, 4, 640, 640, 128, 5, 1, False),     # odd batch and R
]


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: "x".join(map(str, c)))
def test_sharded_small_all_rows(m, cfg):
    B, Hq, Hkv, Sq, Skv, d, R, shift, causal = cfg
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, d, seed=sum(cfg[:7]))
    out, lse = run_sharded(m, q, k, v, R, shift, causal)
    o_ref, l_ref = oracle.attn(q, k, v, causal)
    assert_close(out, lse, o_ref, l_ref, "sharded")


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: "x".join(map(str, c)))
def test_partial_small_all_rows(m, cfg):
    B, Hq, Hkv, Sq, Skv, d, R, shift, causal = cfg
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, d, seed=sum(cfg[:7]) + 1)
    op, lp, out, lse = run_partial_merge(m, q, k, v, R, shift, causal)
    op_ref, lp_ref = oracle.attn_partial(q, k, v, R, shift, causal)
    assert_close(op, lp, op_ref, lp_ref, "partials")
    o_ref, l_ref = oracle.attn(q, k, v, causal)
    assert_close(out, lse, o_ref, l_ref, "partial+merge")


@pytest.mark.parametrize("groups", [1, 2, 3, 8])
@pytest.mark.parametrize("cfg", [(1, 8, 1, 128, 4096, 128, 8, 1, False),
                                 (1, 4, 2, 512, 1024, 64, 8, 4, True),
                                 (2, 2, 2, 384, 384, 128, 3, 1, True)],
                         ids=lambda c: "x".join(map(str, c)))
def test_sharded_split_runs_match_oracle(m, monkeypatch, cfg, groups):
    """mercury_attn_sharded with the shifted step sequence cut into runs
    (split-KV through library scratch + merge) equals plain attention."""
    B, Hq, Hkv, Sq, Skv, d, R, shift, causal = cfg
    monkeypatch.setenv("MERCURY_SPLIT_GROUPS", str(groups))
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, d, seed=sum(cfg[:7]) + groups)
    out, lse = run_sharded(m, q, k, v, R, shift, causal)
    o_ref, l_ref = oracle.attn(q, k, v, causal)
    assert_close(out, lse, o_ref, l_ref, "split into %d runs" % groups)


def test_sharded_auto_split_on_long_kv(m):
    """A short query side over a long KV: the chooser splits (the GPU would
    otherwise hold 16 work items for its SMs); result equals plain attention."""
    info = m.mercury_work_decomposition(1, 8, 1, 512, 65536, 128, 16, False, 0)
    assert info["n_items"] < 8 * torch.cuda.get_device_properties(0).multi_processor_count
    q, k, v = make_qkv(1, 8, 1, 512, 65536, 128, seed=77)
    out, lse = run_sharded(m, q, k, v, 16, 1, False)
    o_ref, l_ref = oracle.attn(q, k, v, False)
    assert_close(out, lse, o_ref, l_ref, "auto split")


@pytest.mark.parametrize("cfg", [
    # B, Hq, Hkv, Sq, Skv, d, n_splits, causal
    (2, 64, 8, 1, 32768, 128, 0, False),     # Llama-3-70B-like decode step, auto split
    (1, 32, 32, 4, 8192, 128, 8, False),     # MHA, 4 queries
    (1, 8, 2, 16, 4096, 64, 0, True),        # causal chunk at the end of the context
    (1, 8, 1, 3, 3000, 128, 3, True),        # odd lengths, 3 splits
    (2, 4, 4, 1, 256, 128, 1, False),        # no split (fused)
], ids=lambda c: "x".join(map(str, c)))
def test_decode_matches_oracle(m, cfg):
    B, Hq, Hkv, Sq, Skv, d, n_splits, causal = cfg
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, d, seed=sum(cfg[:6]))
    out, lse = m.mercury_attn_decode(q.cuda(), k.cuda(), v.cuda(), n_splits, causal)
    m.mercury_sync_status()
    o_ref, l_ref = oracle.attn(q, k, v, causal)
    assert_close(out.cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, "decode")


@pytest.mark.parametrize("cfg", [(1, 4, 4, 512, 512, 64, 4, 1, False), (1, 8, 2, 1024, 1024, 128, 8, 4, True),
                                 (1, 8, 1, 128, 4096, 128, 4, 1, False)], ids=lambda c: "x".join(map(str, c)))
@pytest.mark.parametrize("groups", [1, 4], ids=["fused", "split4"])
def test_sharded_bf16_output(m, cfg, groups, monkeypatch):
    """bf16 O: within the parity tolerance of the oracle, and equal to the fp32
    call's O rounded to bf16 under the same schedule (fused, or cut into runs
    whose fp32 partials are merged before the rounding)."""
    monkeypatch.setenv("MERCURY_SPLIT_GROUPS", str(groups))
    B, Hq, Hkv, Sq, Skv, d, R, shift, causal = cfg
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, d, seed=sum(cfg[:7]) + 99)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o16, l16 = m.mercury_attn_sharded_bf16(qd, kd, vd, R, shift, causal)
    o32, l32 = m.mercury_attn_sharded(qd, kd, vd, R, shift, causal)
    m.mercury_sync_status()
    assert o16.dtype == torch.bfloat16
    assert torch.equal(o16, o32.to(torch.bfloat16))
    assert torch.equal(l16, l32)
    o_ref, l_ref = oracle.attn(q, k, v, causal)
    assert_close(o16.float().cpu().numpy(), l16.cpu().numpy(), o_ref, l_ref, "bf16 out")


# Causal shapes with more work items than the GPU has SMs: each CTA claims its
# next item from the launch's counter when it is free (dynamic scheduling).
DYNAMIC = [
    # B, Hq, Hkv, Sq, Skv, d, R, shift, causal
    (1, 32, 8, 4096, 4096, 128, 8, 1, True),    # 512 items
    (2, 16, 16, 2048, 2048, 64, 4, 2, True),    # MHA row pairs, nested 2x2, 256 items
]


@pytest.mark.parametrize("cfg", DYNAMIC, ids=lambda c: "x".join(map(str, c)))
def test_dynamic_items_all_rows(m, cfg):
    B, Hq, Hkv, Sq, Skv, d, R, shift, causal = cfg
    info = m.mercury_work_decomposition(B, Hq, Hkv, Sq, Skv, d, R, causal, 0)
    assert info["n_items"] > torch.cuda.get_device_properties(0).multi_processor_count
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, d, seed=sum(cfg[:7]) + 3)
    o_ref, l_ref = oracle.attn(q, k, v, causal)
    out, lse = run_sharded(m, q, k, v, R, shift, causal)
    assert_close(out, lse, o_ref, l_ref, "fused, dynamic items")
    _, _, out, lse = run_partial_merge(m, q, k, v, R, shift, causal)
    assert_close(out, lse, o_ref, l_ref, "per-step partials, dynamic items")


def test_dynamic_items_on_two_streams_at_once(m):
    """Two causal calls in flight on two streams take different work-item
    counters: both results are right."""
    cfg = (1, 32, 8, 4096, 4096, 128, 8, 1, True)
    B, Hq, Hkv, Sq, Skv, d, R, shift, causal = cfg
    ins = [make_qkv(B, Hq, Hkv, Sq, Skv, d, seed=s) for s in (71, 72)]
    dev = [tuple(x.cuda() for x in t) for t in ins]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    torch.cuda.synchronize()
    for (qd, kd, vd), st in zip(dev, streams):
        out = torch.empty((B, Hq, Sq, d), device="cuda")
        lse = torch.empty((B, Hq, Sq), device="cuda")
        m.mercury_attn_sharded(qd, kd, vd, R, shift, causal, out, lse, stream=st)
        outs.append((out, lse))
    torch.cuda.synchronize()
    m.mercury_sync_status()
    for (q, k, v), (out, lse) in zip(ins, outs):
        o_ref, l_ref = oracle.attn(q, k, v, causal)
        assert_close(out.cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, "concurrent stream")


@pytest.mark.parametrize("cfg", [(1, 8, 2, 2048, 2048, 128, 4, 1, True),     # fused schedule
                                 (1, 8, 1, 128, 16384, 128, 8, 1, False),   # split-KV + merge
                                 (1, 32, 8, 4096, 4096, 128, 8, 1, True)],  # dynamic work items
                         ids=["fused", "split", "dynamic"])
def test_cuda_graph_capture_and_replay(m, cfg):
    """The calls are stream-ordered and capturable: capture once (after a
    warm-up call on the same stream), replay with new inputs copied in place."""
    B, Hq, Hkv, Sq, Skv, d, R, shift, causal = cfg
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, d, seed=31)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out = torch.empty((B, Hq, Sq, d), device="cuda")
    lse = torch.empty((B, Hq, Sq), device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        m.mercury_attn_sharded(qd, kd, vd, R, shift, causal, out, lse, stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        m.mercury_attn_sharded(qd, kd, vd, R, shift, causal, out, lse, stream=s)
    for seed in (32, 33):
        q2, k2, v2 = make_qkv(B, Hq, Hkv, Sq, Skv, d, seed=seed)
        qd.copy_(q2)
        kd.copy_(k2)
        vd.copy_(v2)
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        m.mercury_sync_status()
        o_ref, l_ref = oracle.attn(q2, k2, v2, causal)
        assert_close(out.cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, "graph replay")


def _scores_that_jump(B, H, Sq, Skv, d, seed):
    """Keys in the second half of the sequence score 12x higher: a rank whose
    shifted order visits a low shard first meets a running max that grows by
    far more than 2^8 (log2 units) at a later tile."""
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, Sq, d, generator=g).bfloat16()
    k = torch.randn(B, H, Skv, d, generator=g)
    k[:, :, Skv // 2:] *= 12.0
    v = torch.randn(B, H, Skv, d, generator=g).bfloat16()
    return q, k.bfloat16(), v


def _sum_above_threshold(B, H, Sq, Skv, d, seed):
    """Every key of the second half scores 2.04 (log2 units) above every key of
    the first: a later tile's probabilities are all ~4.1 relative to the running
    max, so their sum passes 2^8 while the max moves by far less than 2^8."""
    g = torch.Generator().manual_seed(seed)
    q = torch.zeros(B, H, Sq, d)
    q[..., 0] = 8.0
    k = torch.zeros(B, H, Skv, d)
    k[..., 0] = 1.0
    k[:, :, Skv // 2:, 0] = 3.0
    v = torch.randn(B, H, Skv, d, generator=g).bfloat16()
    return q.bfloat16(), k.bfloat16(), v


@pytest.mark.parametrize("make", [_scores_that_jump, _sum_above_threshold], ids=["max_jump", "sum_over_2e8"])
@pytest.mark.parametrize("causal", [False, True])
def test_running_max_paths(m, make, causal):
    """The softmax takes the exponentials with the running max first and redoes a
    tile only when its probabilities could exceed 2^8: both redo cases (the max
    moves, and it does not) must give plain attention, fused and per step."""
    B, H, Sq, Skv, d, R = 1, 2, 1024, 1024, 128, 4
    q, k, v = make(B, H, Sq, Skv, d, seed=21)
    o_ref, l_ref = oracle.attn(q, k, v, causal)
    out, lse = run_sharded(m, q, k, v, R, 1, causal)
    assert_close(out, lse, o_ref, l_ref, "fused")
    _, _, out, lse = run_partial_merge(m, q, k, v, R, 1, causal)
    assert_close(out, lse, o_ref, l_ref, "partial + merge")


def test_shift_orders_agree_on_gpu(m):
    q, k, v = make_qkv(1, 4, 2, 1024, 1024, 128, seed=42)
    o_ref, l_ref = oracle.attn(q, k, v, True)
    for shift in (0, 1, 2, 4, 8):
        out, lse = run_sharded(m, q, k, v, 8, shift, True)
        assert_close(out, lse, o_ref, l_ref, "shift %d" % shift)


def test_deterministic_replay(m):
    q, k, v = make_qkv(1, 8, 2, 2048, 2048, 128, seed=9)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = m.mercury_attn_sharded(qd, kd, vd, 4, 1, True)
    o2, l2 = m.mercury_attn_sharded(qd, kd, vd, 4, 1, True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_output_canaries_untouched(m):
    B, Hq, Hkv, S, d, R = 1, 4, 2, 320, 128, 2
    q, k, v = make_qkv(B, Hq, Hkv, S, S, d, seed=3)
    n_o, n_l = B * Hq * S * d, B * Hq * S
    big_o = torch.full((n_o + 4096,), 7.25, device="cuda")
    big_l = torch.full((n_l + 4096,), 7.25, device="cuda")
    out = big_o[:n_o].view(B, Hq, S, d)
    lse = big_l[:n_l].view(B, Hq, S)
    m.mercury_attn_sharded(q.cuda(), k.cuda(), v.cuda(), R, 1, True, out=out, lse=lse)
    torch.cuda.synchronize()
    assert (big_o[n_o:] == 7.25).all() and (big_l[n_l:] == 7.25).all()


def _guarded(n, dtype, fill=7.25, pad=4096):
    """A buffer of n elements with `pad` canary elements on each side."""
    big = torch.full((n + 2 * pad,), fill, dtype=dtype, device="cuda")
    return big, big[pad:pad + n]


def _canaries_intact(big, n, fill=7.25, pad=4096):
    return bool((big[:pad] == fill).all()) and bool((big[pad + n:] == fill).all())


@pytest.mark.parametrize("cfg", [(1, 4, 2, 320, 320, 128, 2, 1, True), (1, 8, 1, 96, 3072, 64, 3, 1, False)],
                         ids=["gqa_causal", "mqa_packed"])
def test_partial_and_merge_canaries_untouched(m, cfg):
    """Per-step partials (every slot) and the merge's outputs are written
    inside their arrays only: canaries on both sides stay intact."""
    B, Hq, Hkv, Sq, Skv, d, R, shift, causal = cfg
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, d, seed=17)
    rows = B * Hq * Sq
    bo, op = _guarded(R * rows * d, torch.float32)
    bl, lp = _guarded(R * rows, torch.float32)
    m.mercury_attn_partial(q.cuda(), k.cuda(), v.cuda(), R, shift, causal, op.view(R, B, Hq, Sq, d),
                           lp.view(R, B, Hq, Sq))
    bmo, mo = _guarded(rows * d, torch.float32)
    bml, ml = _guarded(rows, torch.float32)
    m.mercury_lse_merge(op.view(R, B, Hq, Sq, d), lp.view(R, B, Hq, Sq), mo.view(B, Hq, Sq, d), ml.view(B, Hq, Sq))
    m.mercury_sync_status()
    assert _canaries_intact(bo, R * rows * d) and _canaries_intact(bl, R * rows)
    assert _canaries_intact(bmo, rows * d) and _canaries_intact(bml, rows)
    o_ref, l_ref = oracle.attn(q, k, v, causal)
    assert_close(mo.cpu().numpy(), ml.cpu().numpy(), o_ref, l_ref, "merge inside canaries")


@pytest.mark.parametrize("groups", [1, 3], ids=["fused", "split3"])
def test_bf16_output_canaries_untouched(m, groups, monkeypatch):
    """bf16 O (fused, or split runs merged then rounded) stays inside its array."""
    monkeypatch.setenv("MERCURY_SPLIT_GROUPS", str(groups))
    B, Hq, Hkv, S, d, R = 1, 4, 2, 384, 128, 3
    q, k, v = make_qkv(B, Hq, Hkv, S, S, d, seed=19)
    n_o, n_l = B * Hq * S * d, B * Hq * S
    bo, out = _guarded(n_o, torch.bfloat16)
    bl, lse = _guarded(n_l, torch.float32)
    m.mercury_attn_sharded_bf16(q.cuda(), k.cuda(), v.cuda(), R, 1, True, out.view(B, Hq, S, d),
                                lse.view(B, Hq, S))
    m.mercury_sync_status()
    assert _canaries_intact(bo, n_o) and _canaries_intact(bl, n_l)
    o_ref, l_ref = oracle.attn(q, k, v, True)
    assert_close(out.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, "bf16 inside canaries")


@pytest.mark.parametrize("bf16", [False, True], ids=["fp32_out", "bf16_out"])
def test_output_16_byte_aligned_only(m, bf16, monkeypatch):
    """O at an address that is 16- but not 32-byte aligned takes the 16-byte
    store path: bit-identical to the 32-byte path, canaries around it intact."""
    monkeypatch.setenv("MERCURY_SPLIT_GROUPS", "1")
    B, Hq, Hkv, S, d, R = 1, 4, 2, 512, 128, 4
    q, k, v = (x.cuda() for x in make_qkv(B, Hq, Hkv, S, S, d, seed=13))
    dt = torch.bfloat16 if bf16 else torch.float32
    fn = m.mercury_attn_sharded_bf16 if bf16 else m.mercury_attn_sharded
    n_o = B * Hq * S * d
    shift = 16 // torch.tensor([], dtype=dt).element_size()  # 16 bytes
    big = torch.full((n_o + 2 * shift + 64,), 3.5, dtype=dt, device="cuda")
    assert big.data_ptr() % 256 == 0
    out = big[shift:shift + n_o].view(B, Hq, S, d)
    assert out.data_ptr() % 32 == 16
    o_ref = torch.empty((B, Hq, S, d), dtype=dt, device="cuda")
    l_ref = torch.empty((B, Hq, S), device="cuda")
    lse = torch.empty((B, Hq, S), device="cuda")
    fn(q, k, v, R, 1, True, out, lse)
    fn(q, k, v, R, 1, True, o_ref, l_ref)
    m.mercury_sync_status()
    assert torch.equal(out, o_ref) and torch.equal(lse, l_ref)
    assert (big[:shift] == 3.5).all() and (big[shift + n_o:] == 3.5).all()


# ------------------------------------------------------ merge kernel

@pytest.mark.parametrize("n_parts,rows,d", [(1, 7, 128), (4, 33, 64), (64, 1000, 128),
                                            (3, 5, 4), (130, 17, 256), (8, 64, 12), (4096, 3, 128),
                                            (2, 1, 512)])
def test_lse_merge_matches_oracle(m, n_parts, rows, d):
    g = torch.Generator().manual_seed(n_parts * 1000 + rows)
    o = torch.randn(n_parts, rows, d, generator=g)
    l = torch.randn(n_parts, rows, generator=g) * 4
    l[:, 0] = -math.inf                     # a row with no contribution at all
    if n_parts > 1:
        l[0, 1:] = -math.inf                # masked parts
        o[0, 1:] = 0.0
    out, lse = m.mercury_lse_merge(o.cuda(), l.cuda())
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.lse_merge(o.double().numpy(), l.double().numpy())
    fin = np.isfinite(l_ref)
    assert (np.isfinite(lse.cpu().numpy()) == fin).all()
    np.testing.assert_allclose(out.cpu().numpy(), o_ref, atol=1e-5, rtol=1e-5)
    np.testing.assert_allclose(lse.cpu().numpy()[fin], l_ref[fin], atol=1e-5, rtol=0)


# ------------------------------------------------------ fault path (no GPU fault)

@pytest.mark.parametrize("fault", ["drop_p_arrive", "drop_kv_free"])
def test_bounded_wait_times_out_cleanly(m, monkeypatch, fault):
    """A dropped arrive makes a device wait run out: the kernel records
    ETIMEOUT and returns; the context stays usable for the next call.
    drop_p_arrive starves the MMA issuer; drop_kv_free starves the TMA
    producer after it has issued loads, so its exit path (wait for the loads
    it issued to land) runs too."""
    q, k, v = make_qkv(1, 2, 1, 512, 512, 128, seed=1)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    monkeypatch.setenv("MERCURY_FAULT", fault)
    monkeypatch.setenv("MERCURY_WAIT_NS", "20000000")
    m.mercury_attn_sharded(qd, kd, vd, 2, 1, False)
    with pytest.raises(m.MercuryError) as e:
        m.mercury_sync_status()
    assert e.value.status == m.MERCURY_ETIMEOUT
    assert "site 0x" in str(e.value)
    monkeypatch.delenv("MERCURY_FAULT")
    monkeypatch.delenv("MERCURY_WAIT_NS")
    out, lse = m.mercury_attn_sharded(qd, kd, vd, 2, 1, False)
    m.mercury_sync_status()
    o_ref, l_ref = oracle.attn(q, k, v, False)
    assert_close(out.cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, "after timeout")


def test_sync_check_env_reports_timeout(m, monkeypatch):
    q, k, v = make_qkv(1, 2, 1, 256, 256, 64, seed=2)
    monkeypatch.setenv("MERCURY_FAULT", "drop_p_arrive")
    monkeypatch.setenv("MERCURY_WAIT_NS", "20000000")
    monkeypatch.setenv("MERCURY_SYNC_CHECK", "1")
    with pytest.raises(m.MercuryError) as e:
        m.mercury_attn_sharded(q.cuda(), k.cuda(), v.cuda(), 1, 1, False)
    assert e.value.status == m.MERCURY_ETIMEOUT
    monkeypatch.delenv("MERCURY_FAULT")
    m.mercury_attn_sharded(q.cuda(), k.cuda(), v.cuda(), 1, 1, False)


# ------------------------------------------------------ full-size workloads

def _run_workload(m, name, check_cross=True):
    w = WORKLOADS[name]
    B, Hq, Hkv, Sq, Skv, d = w["B"], w["Hq"], w["Hkv"], w["Sq"], w["Skv"], w["d"]
    R, shift, causal = w["R"], w["shift"], w["causal"]
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, d, seed=w["seed"], scale=w["scale"])
    rows = sample_rows(B, Hq, Sq, R, seed=w["seed"], n_heads=8 if B * Hq > 8 else B * Hq)
    o_ref, l_ref = oracle.attn(q, k, v, causal, rows=rows)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    del q, k, v
    if w["mode"] == "partial":
        op, lp = m.mercury_attn_partial(qd, kd, vd, R, shift, causal)
        out, lse = m.mercury_lse_merge(op, lp)
        del op, lp
    else:
        out, lse = m.mercury_attn_sharded(qd, kd, vd, R, shift, causal)
    m.mercury_sync_status()
    ridx = torch.as_tensor(rows, device="cuda")
    o_s = out.view(-1, d)[ridx].cpu().numpy()
    l_s = lse.view(-1)[ridx].cpu().numpy()
    assert_close(o_s, l_s, o_ref, l_ref, name + " sampled rows")
    if check_cross:
        # every row: fused vs partial + merge on the GPU
        if w["mode"] == "partial":
            o2, l2 = m.mercury_attn_sharded(qd, kd, vd, R, shift, causal)
        else:
            op, lp = m.mercury_attn_partial(qd, kd, vd, R, shift, causal)
            o2, l2 = m.mercury_lse_merge(op, lp)
            del op, lp
        m.mercury_sync_status()
        diff = (o2 - out).abs()
        assert diff.max().item() <= O_MAX and diff.mean().item() <= O_MEAN
        assert (l2 - lse).abs().max().item() <= LSE_MAX
    del out, lse, qd, kd, vd
    torch.cuda.empty_cache()


def test_workload_mha_b1_h4_d64_s512_r4(m):
    _run_workload(m, "mha_b1_h4_d64_s512_r4")


def test_workload_gqa_32k_causal(m):
    _run_workload(m, "gqa_b1_hq32_hkv8_d128_s32k_causal_r8")


def test_workload_mha_b16_4k(m):
    _run_workload(m, "mha_b16_h32_d128_s4k_r8")


def test_workload_mqa_2m_merge(m):
    _run_workload(m, "mqa_b1_hq8_hkv1_d128_sq2k_skv2m_r64_merge")


@pytest.mark.slow
def test_workload_gqa_128k_causal_nested(m):
    _run_workload(m, "gqa_b1_hq64_hkv8_d128_s128k_causal_r8_nested2x4", check_cross=True)


# ------------------------------------------------------ randomised shapes

def _random_shapes(n, seed):
    """Seeded shapes within the call's contract: d 64 or 128, GQA group 1-8,
    R dividing both lengths, lengths that are not multiples of the 128-row
    tiles, causal only with Sq <= Skv, every shift form R admits."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        d = int(rng.choice([64, 128]))
        Hkv = int(rng.choice([1, 2, 3]))
        G = int(rng.choice([1, 2, 4, 8]))
        B = int(rng.choice([1, 2]))
        R = int(rng.choice([1, 2, 3, 4, 6, 8]))
        Sq = R * int(rng.integers(8, 160))
        Skv = Sq if rng.random() < 0.5 else R * int(rng.integers(8, 320))
        causal = bool(rng.random() < 0.5) and Sq <= Skv
        shifts = [0, 1] + [k for k in range(2, R) if R % k == 0]
        shift = int(rng.choice(shifts))
        out.append((B, Hkv * G, Hkv, Sq, Skv, d, R, shift, causal))
    return out


@pytest.mark.parametrize("cfg", _random_shapes(12, 2026), ids=lambda c: "x".join(map(str, c)))
def test_random_shapes_all_paths(m, cfg):
    """Fused, per-step partials + merge and bf16 O on a seeded random shape,
    every row against the oracle."""
    B, Hq, Hkv, Sq, Skv, d, R, shift, causal = cfg
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, d, seed=sum(cfg[:7]) + 11)
    o_ref, l_ref = oracle.attn(q, k, v, causal)
    out, lse = run_sharded(m, q, k, v, R, shift, causal)
    assert_close(out, lse, o_ref, l_ref, "fused")
    _, _, out, lse = run_partial_merge(m, q, k, v, R, shift, causal)
    assert_close(out, lse, o_ref, l_ref, "partials + merge")
    o16, l16 = m.mercury_attn_sharded_bf16(q.cuda(), k.cuda(), v.cuda(), R, shift, causal)
    m.mercury_sync_status()
    assert_close(o16.float().cpu().numpy(), l16.cpu().numpy(), o_ref, l_ref, "bf16 O")


# ---------------------------------------- shift-table capacity (R <= 32 / R > 32)

@pytest.mark.parametrize("cfg", [
    # B, Hq, Hkv, Sq, Skv, d, R, shift, causal
    (1, 4, 2, 31 * 24, 31 * 24, 128, 31, 1, True),    # prime R: flat or unshifted only
    (1, 4, 2, 31 * 16, 31 * 40, 64, 31, 0, False),
    (1, 4, 4, 32 * 24, 32 * 24, 64, 32, 8, True),     # the small table's last R, nested 4 x 8
    (1, 4, 1, 32 * 16, 32 * 48, 128, 32, 1, False),
    (1, 4, 2, 33 * 24, 33 * 24, 128, 33, 11, True),   # the large table's first R, nested 3 x 11
    (2, 2, 2, 33 * 16, 33 * 16, 64, 33, 1, False),
    (1, 8, 2, 48 * 16, 48 * 16, 128, 48, 6, True),    # nested 8 x 6
    (1, 4, 1, 64 * 8, 64 * 32, 64, 64, 16, False),    # nested 4 x 16
], ids=lambda c: "x".join(map(str, c)))
def test_shift_table_capacity_boundary(m, cfg, monkeypatch):
    """Calls with R <= 32 carry a 32 x 32 shift table in the kernel
    parameters, larger R the full one: on both sides of the switch the fused
    path, the per-step partials (each slot against the oracle's) and a split
    into runs equal plain attention on every row."""
    B, Hq, Hkv, Sq, Skv, d, R, shift, causal = cfg
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, d, seed=sum(cfg[:7]) + 29)
    o_ref, l_ref = oracle.attn(q, k, v, causal)
    out, lse = run_sharded(m, q, k, v, R, shift, causal)
    assert_close(out, lse, o_ref, l_ref, "fused")
    op, lp, out, lse = run_partial_merge(m, q, k, v, R, shift, causal)
    op_ref, lp_ref = oracle.attn_partial(q, k, v, R, shift, causal)
    assert_close(op, lp, op_ref, lp_ref, "partials")
    assert_close(out, lse, o_ref, l_ref, "partials + merge")
    monkeypatch.setenv("MERCURY_SPLIT_GROUPS", "3")
    out, lse = run_sharded(m, q, k, v, R, shift, causal)
    assert_close(out, lse, o_ref, l_ref, "split into 3 runs")


def _random_large_r_shapes(n, seed):
    """Seeded shapes with many virtual ranks (R from 12 to 96, on both sides
    of the shift table's 32-rank capacity): short blocks and shards, every
    shift form R admits, GQA groups, causal only with Sq <= Skv."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        R = int(rng.choice([12, 16, 24, 40, 48, 56, 64, 80, 96]))
        d = int(rng.choice([64, 128]))
        Hkv = int(rng.choice([1, 2]))
        G = int(rng.choice([1, 2, 4]))
        Sq = R * int(rng.integers(2, 24))
        Skv = Sq if rng.random() < 0.5 else R * int(rng.integers(2, 48))
        causal = bool(rng.random() < 0.5) and Sq <= Skv
        shifts = [0, 1] + [k for k in range(2, R) if R % k == 0]
        shift = int(rng.choice(shifts))
        out.append((1, Hkv * G, Hkv, Sq, Skv, d, R, shift, causal))
    return out


@pytest.mark.parametrize("cfg", _random_large_r_shapes(10, 2027), ids=lambda c: "x".join(map(str, c)))
def test_random_large_r_all_paths(m, cfg, monkeypatch):
    """Fused, per-step partials + merge and a split into runs on a seeded
    shape with many virtual ranks, every row against the oracle."""
    B, Hq, Hkv, Sq, Skv, d, R, shift, causal = cfg
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, d, seed=sum(cfg[:7]) + 17)
    o_ref, l_ref = oracle.attn(q, k, v, causal)
    out, lse = run_sharded(m, q, k, v, R, shift, causal)
    assert_close(out, lse, o_ref, l_ref, "fused")
    _, _, out, lse = run_partial_merge(m, q, k, v, R, shift, causal)
    assert_close(out, lse, o_ref, l_ref, "partials + merge")
    monkeypatch.setenv("MERCURY_SPLIT_GROUPS", "5")
    out, lse = run_sharded(m, q, k, v, R, shift, causal)
    assert_close(out, lse, o_ref, l_ref, "split into 5 runs")
