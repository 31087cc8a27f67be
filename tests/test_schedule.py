"""Schedule selection under a device-memory budget: the static filter, the
cost estimate and, on a GPU, running / tuning / measuring schedules.

CPU tests pin the planner's arithmetic against an independent brute force:
every candidate's memory is recomputed from the tensor sizes, its predicted
time from a round-robin simulation over the work items that
mercury_work_item_rows reports (key tiles counted from the oracle's own shift
table and the causal limit), and the Pareto flags by pairwise comparison.
GPU tests check that every candidate schedule computes plain attention (the
oracle) and that tuning picks, caches and re-checks a schedule."""
import ctypes
import math

import numpy as np
import pytest

from long_context_sharded_gb300.inputs import make_qkv


@pytest.fixture(scope="module")
def m():
    from long_context_sharded_gb300 import build
    build.build()
    from long_context_sharded_gb300 import mercury
    return mercury


def profile(m, **kw):
    p = m.CostProfile()
    vals = dict(tile_us=1.0, tile1_us=1.0, item_us=3.0, launch_us=5.0, merge_gbs=1000.0,
                hbm_gbs=1e9, n_sms=7, measured=0)
    vals.update(kw)
    for k, v in vals.items():
        setattr(p, k, v)
    return p


def io_bytes(B, Hq, Hkv, Sq, Skv, d):
    return B * Hq * Sq * d * 2 + 2 * B * Hkv * Skv * d * 2 + B * Hq * Sq * d * 4 + B * Hq * Sq * 4


def distinct_runs(R):
    out = []
    for g in range(1, R + 1):
        spg = -(-R // g)
        if -(-R // spg) == g:
            out.append(g)
    return out


# ------------------------------------------------------------------ CPU


def test_default_profile(m):
    p = m.mercury_default_cost_profile(152)
    assert p.n_sms == 152 and p.measured == 0
    for f in ("tile_us", "tile1_us", "item_us", "launch_us", "merge_gbs", "hbm_gbs"):
        assert getattr(p, f) > 0, f
    assert p.tile1_us < p.tile_us
    rc = m.lib.mercury_default_cost_profile(0, ctypes.byref(m.CostProfile()))
    assert rc == m.MERCURY_EINVAL


SHAPES = [
    # B, Hq, Hkv, Sq, Skv, d, causal, R, shift
    (1, 4, 2, 512, 1024, 64, True, 8, 4),
    (2, 2, 2, 384, 384, 128, True, 3, 1),
    (1, 8, 1, 128, 4096, 128, False, 8, 1),
    (1, 6, 2, 256, 512, 64, True, 4, 0),     # three head tiles per KV group: odd head pairs
    (1, 32, 8, 2048, 2048, 128, True, 8, 1), # causal, more items than SMs: claimed dynamically
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_candidates_memory_and_count(m, shape):
    B, Hq, Hkv, Sq, Skv, d, causal, R, shift = shape
    plans, n = m.mercury_plan_schedules(B, Hq, Hkv, Sq, Skv, d, causal, R, shift, 0, profile(m))
    rq_options = [R] + ([1] if R > 1 else [])
    expect = {(R, rq, g) for rq in rq_options if Sq % rq == 0 for g in distinct_runs(R)}
    assert n == len(plans) == len(expect)
    assert {(p.R, p.Rq, p.n_runs) for p in plans} == expect
    io = io_bytes(B, Hq, Hkv, Sq, Skv, d)
    for p in plans:
        scratch = 0 if p.n_runs == 1 else p.n_runs * B * Hq * Sq * (d + 1) * 4
        assert p.scratch_bytes == scratch
        assert p.hbm_bytes == io + scratch
        assert p.shift == shift and p.measured_us == -1.0
        if p.Rq == p.R:
            mode = 0 if p.n_runs == 1 else (1 if p.n_runs == p.R else p.n_runs)
            info = m.mercury_work_decomposition(B, Hq, Hkv, Sq, Skv, d, R, causal, mode)
            assert p.work_items == info["n_items"]
    t = [p.predicted_us for p in plans]
    assert t == sorted(t)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_budget_filter_and_pareto(m, shape):
    B, Hq, Hkv, Sq, Skv, d, causal, R, shift = shape
    prof = profile(m)
    all_plans, n_all = m.mercury_plan_schedules(B, Hq, Hkv, Sq, Skv, d, causal, R, shift, 0, prof)
    # Pareto: nothing else is no larger and no slower, and better in one
    for a in all_plans:
        dominated = any(b.hbm_bytes <= a.hbm_bytes and b.predicted_us <= a.predicted_us and
                        (b.hbm_bytes < a.hbm_bytes or b.predicted_us < a.predicted_us)
                        for b in all_plans)
        assert a.pareto == (0 if dominated else 1)
    io = io_bytes(B, Hq, Hkv, Sq, Skv, d)
    sizes = sorted({p.hbm_bytes for p in all_plans})
    for budget in sizes:
        plans, n = m.mercury_plan_schedules(B, Hq, Hkv, Sq, Skv, d, causal, R, shift, budget, prof)
        assert n == sum(1 for p in all_plans if p.hbm_bytes <= budget)
        assert all(p.hbm_bytes <= budget for p in plans)
    with pytest.raises(m.MercuryError) as e:
        m.mercury_plan_schedules(B, Hq, Hkv, Sq, Skv, d, causal, R, shift, io - 1, prof)
    assert e.value.status == m.MERCURY_EBUDGET
    assert str(io) in str(e.value)
    # the fused schedule needs no scratch: a budget of exactly the tensors admits it
    plans, _ = m.mercury_plan_schedules(B, Hq, Hkv, Sq, Skv, d, causal, R, shift, io, prof)
    assert plans and all(p.n_runs == 1 for p in plans)


def simulate(m, oracle, shape, runs, prof):
    """Simulation of one candidate with Rq = R, item by item: round robin, or,
    for a causal launch with more items than CTAs, each item to the CTA that
    is free earliest (the kernel claims items dynamically there)."""
    import heapq
    B, Hq, Hkv, Sq, Skv, d, causal, R, shift = shape
    mode = 0 if runs == 1 else (1 if runs == R else runs)
    info = m.mercury_work_decomposition(B, Hq, Hkv, Sq, Skv, d, R, causal, mode)
    n_items = info["n_items"]
    order = oracle.shift_order(R, shift)
    Bq, Bk = Sq // R, Skv // R
    spg = -(-R // runs)
    grid = min(n_items, prof.n_sms)
    busy = [0.0] * grid
    dynamic = causal and n_items > grid
    heap = [(0.0, c) for c in range(grid)]
    for item in range(n_items):
        rows, slot = m.mercury_work_item_rows(B, Hq, Hkv, Sq, Skv, d, R, shift, causal, mode, item)
        qs = [r % Sq for r in rows]
        ranks = {q // Bq for q in qs}
        assert len(ranks) == 1
        rank = ranks.pop()
        kv_end = min(Skv, max(qs) + Skv - Sq + 1) if causal else Skv
        if mode == 0:
            steps = range(R)
        elif mode == 1:
            steps = [slot]
        else:
            steps = range(slot * spg, min(R, (slot + 1) * spg))
        tiles = 0
        for j in steps:
            s = order[rank][j]
            lo, hi = s * Bk, min(s * Bk + Bk, kv_end)
            tiles += max(0, -(-(hi - lo) // 128))
        cost = prof.item_us + tiles * prof.tile_us
        if dynamic:
            until, cta = heapq.heappop(heap)
            heapq.heappush(heap, (until + cost, cta))
            busy[cta] = until + cost
        else:
            busy[item % grid] += cost
    t = prof.launch_us + max(busy)
    if runs > 1:
        rows_total = B * Hq * Sq
        t += prof.launch_us + (runs + 1) * rows_total * (d + 1) * 4 / (prof.merge_gbs * 1e3)
    return t


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_predicted_time_matches_brute_force(m, shape):
    import oracle
    B, Hq, Hkv, Sq, Skv, d, causal, R, shift = shape
    prof = profile(m)
    plans, _ = m.mercury_plan_schedules(B, Hq, Hkv, Sq, Skv, d, causal, R, shift, 0, prof)
    checked = 0
    for p in plans:
        if p.Rq != p.R:
            continue
        want = simulate(m, oracle, shape, p.n_runs, prof)
        assert math.isclose(p.predicted_us, want, rel_tol=1e-9), (p.n_runs, p.predicted_us, want)
        checked += 1
    assert checked == len(distinct_runs(R))


def test_closed_forms(m):
    n = 5
    prof = profile(m, n_sms=n, tile_us=2.0, tile1_us=0.75, item_us=3.0, launch_us=4.0)

    def fused(Hq, Sq, Skv, **kw):
        p = profile(m, n_sms=n, tile_us=2.0, tile1_us=0.75, item_us=3.0, launch_us=4.0, **kw)
        plans, _ = m.mercury_plan_schedules(1, Hq, Hq, Sq, Skv, 128, False, 1, 0, 0, p)
        assert len(plans) == 1 and plans[0].n_runs == 1
        return plans[0]

    # one item per SM, two query tiles of 128 rows, 16 key tiles
    assert fused(n, 256, 2048).predicted_us == pytest.approx(4.0 + 3.0 + 16 * 2.0)
    # two items per SM
    assert fused(2 * n, 256, 2048).predicted_us == pytest.approx(4.0 + 2 * (3.0 + 16 * 2.0))
    # one item more than SMs: the busiest SM runs two
    assert fused(n + 1, 256, 2048).predicted_us == pytest.approx(4.0 + 2 * (3.0 + 16 * 2.0))
    # one query tile per item
    assert fused(n, 128, 8192).predicted_us == pytest.approx(4.0 + 3.0 + 64 * 0.75)
    # memory floor: at 1 GB/s the traffic dominates
    p = fused(n, 256, 2048, hbm_gbs=1.0)
    traffic = n * 256 * 128 * 2 + 2 * n * 2048 * 128 * 2 + n * 256 * 129 * 4
    assert p.predicted_us == pytest.approx(4.0 + traffic / 1e3)
    del prof


CHOOSE_SHAPES = [
    # B, Hq, Hkv, Sq, Skv, d, causal, R, shift
    (1, 32, 8, 32768, 32768, 128, True, 8, 1),
    (1, 64, 8, 131072, 131072, 128, True, 8, 4),
    (16, 32, 32, 4096, 4096, 128, False, 8, 1),
    (1, 8, 1, 2048, 2097152, 128, False, 64, 1),
    (1, 4, 4, 512, 512, 64, False, 4, 1),
    (1, 8, 1, 64, 131072, 128, True, 16, 1),
    (2, 24, 8, 6144, 6144, 64, True, 8, 2),
    (1, 40, 8, 3072, 4096, 128, True, 4, 1),
    (3, 12, 4, 1536, 1536, 128, True, 16, 4),
    (1, 16, 2, 256, 65536, 128, False, 32, 0),
    (4, 8, 8, 1024, 1024, 64, True, 8, 1),
]


@pytest.mark.parametrize("cap", [-1, 0, 200 << 20])
@pytest.mark.parametrize("shape", CHOOSE_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_choose_runs_is_the_planner_argmin(m, shape, cap, monkeypatch):
    """The run count mercury_attn_sharded uses is the planner's fastest Rq = R
    candidate whose scratch fits the cap (ties: fewer runs), although the
    chooser skips candidates by their lower bound instead of estimating all."""
    monkeypatch.delenv("MERCURY_SPLIT_GROUPS", raising=False)
    monkeypatch.delenv("MERCURY_SCRATCH_MAX_BYTES", raising=False)
    B, Hq, Hkv, Sq, Skv, d, causal, R, shift = shape
    prof = m.mercury_default_cost_profile(152)
    plans, _ = m.mercury_plan_schedules(B, Hq, Hkv, Sq, Skv, d, causal, R, shift, 0, prof, 512)
    limit = (4 << 30) if cap < 0 else cap
    fits = [p for p in plans if p.Rq == R and (p.n_runs == 1 or p.scratch_bytes <= limit)]
    best = min(fits, key=lambda p: (p.predicted_us, p.n_runs))
    assert m.mercury_choose_runs(B, Hq, Hkv, Sq, Skv, d, causal, R, shift, 152, cap) == best.n_runs


def test_choose_runs_forced_and_rejects(m, monkeypatch):
    monkeypatch.setenv("MERCURY_SPLIT_GROUPS", "3")
    assert m.mercury_choose_runs(1, 8, 1, 2048, 2097152, 128, False, 64, 1, 152) == 3
    monkeypatch.setenv("MERCURY_SPLIT_GROUPS", "100")
    assert m.mercury_choose_runs(1, 8, 1, 2048, 2097152, 128, False, 64, 1, 152) == 64
    monkeypatch.delenv("MERCURY_SPLIT_GROUPS")
    assert m.mercury_choose_runs(1, 8, 8, 256, 256, 128, False, 1, 1, 152) == 1
    for args in [(1, 8, 3, 256, 256, 128, False, 8, 1, 152), (1, 8, 8, 256, 256, 96, False, 8, 1, 152),
                 (1, 8, 8, 256, 250, 128, False, 8, 1, 152), (1, 8, 8, 256, 256, 128, False, 8, 1, 0),
                 (1, 8, 8, 512, 256, 128, True, 8, 1, 152)]:
        with pytest.raises(m.MercuryError) as e:
            m.mercury_choose_runs(*args)
        assert e.value.status == m.MERCURY_EINVAL
    n = ctypes.c_int(0)
    assert m.lib.mercury_choose_runs(1, 8, 8, 256, 256, 128, 0, 8, 1, 152, -1, None) == m.MERCURY_EINVAL


def test_choose_r(m):
    prof = m.mercury_default_cost_profile(152)
    plans, n = m.mercury_plan_schedules(1, 8, 2, 768, 1536, 128, True, 0, 1, 0, prof)
    assert {p.R for p in plans} == {r for r in range(1, 129) if 1536 % r == 0}
    for p in plans:
        assert p.Rq in (p.R, 1) and 768 % p.Rq == 0
    # nested shift 4: only R that 4 divides
    plans, n = m.mercury_plan_schedules(1, 8, 2, 768, 1536, 128, True, 0, 4, 0, prof)
    assert {p.R for p in plans} == {r for r in range(1, 129) if 1536 % r == 0 and r % 4 == 0}


@pytest.mark.parametrize("kw", [dict(R=5), dict(R=129), dict(R=-1), dict(shift=3), dict(d=96),
                                dict(Hkv=3), dict(causal=True, Sq=2048)])
def test_plan_rejects(m, kw):
    a = dict(B=1, Hq=4, Hkv=2, Sq=256, Skv=1024, d=128, causal=False, R=8, shift=1)
    a.update(kw)
    with pytest.raises(m.MercuryError) as e:
        m.mercury_plan_schedules(a["B"], a["Hq"], a["Hkv"], a["Sq"], a["Skv"], a["d"], a["causal"],
                                 a["R"], a["shift"], 0, m.mercury_default_cost_profile(152))
    assert e.value.status == m.MERCURY_EINVAL


def test_plan_rejects_bad_profile(m):
    n = ctypes.c_int(0)
    for bad in (dict(n_sms=0), dict(tile_us=-1.0), dict(merge_gbs=0.0), dict(hbm_gbs=0.0)):
        rc = m.lib.mercury_plan_schedules(1, 4, 2, 256, 1024, 128, 0, 8, 1, 0,
                                          ctypes.byref(profile(m, **bad)), None, 0, ctypes.byref(n))
        assert rc == m.MERCURY_EINVAL, bad
    rc = m.lib.mercury_plan_schedules(1, 4, 2, 256, 1024, 128, 0, 8, 1, 0, None, None, 0, ctypes.byref(n))
    assert rc == m.MERCURY_EINVAL


P = 0x100000  # fake, aligned "device" address: validation fails before any CUDA call


@pytest.mark.parametrize("tup", [(8, 3, 1, 1), (8, 8, 9, 1), (8, 8, 0, 1), (8, 8, 2, 3), (5, 5, 1, 1),
                                 (0, 1, 1, 1), (129, 1, 1, 1)])
def test_run_schedule_rejects_invalid_tuples(m, tup):
    s = m.Schedule()
    s.R, s.Rq, s.n_runs, s.shift = tup
    rc = m.lib.mercury_attn_run_schedule(P, P, P, 1, 4, 2, 256, 1024, 128, 0, ctypes.byref(s), P, P, None)
    assert rc == m.MERCURY_EINVAL, m.lib.mercury_last_error()


def test_tune_rejects_bad_top_k(m):
    for k in (0, 17):
        rc = m.lib.mercury_tune_schedule(P, P, P, 1, 4, 2, 256, 1024, 128, 8, 1, 0, 0, k, P, P, None,
                                         None, None)
        assert rc == m.MERCURY_EINVAL


# ------------------------------------------------------------------ GPU

O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3


def assert_close(out, lse, o_ref, l_ref, what):
    out = np.asarray(out, dtype=np.float64).reshape(o_ref.shape)
    lse = np.asarray(lse, dtype=np.float64).reshape(l_ref.shape)
    diff = np.abs(out - o_ref)
    assert diff.max() <= O_MAX and diff.mean() <= O_MEAN, (what, diff.max(), diff.mean())
    fin = np.isfinite(l_ref)
    assert (np.isfinite(lse) == fin).all(), what
    assert np.abs(lse[fin] - l_ref[fin]).max() <= LSE_MAX, what


@pytest.fixture(scope="module")
def gpu(m):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return m


GPU_SHAPES = [
    (1, 4, 2, 512, 1024, 64, True, 8, 4),
    (1, 8, 1, 128, 4096, 128, False, 8, 1),
    (2, 6, 2, 96, 1920, 128, True, 6, 1),      # odd head tiles, ragged key tiles, Sq < Skv
    (1, 16, 2, 3, 8192, 128, False, 16, 1),    # decode-like: only Rq = 1 divides Sq
]


@pytest.mark.gpu
@pytest.mark.parametrize("shape", GPU_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_every_candidate_schedule_matches_oracle(gpu, shape):
    import oracle
    m = gpu
    B, Hq, Hkv, Sq, Skv, d, causal, R, shift = shape
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, d, seed=sum(shape[:6]) + 5)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o_ref, l_ref = oracle.attn(q, k, v, causal)
    plans, n = m.mercury_plan_schedules(B, Hq, Hkv, Sq, Skv, d, causal, R, shift, 0,
                                        m.mercury_default_cost_profile(148))
    assert n == len(plans) and n >= 2
    for p in plans:
        out, lse = m.mercury_attn_run_schedule(qd, kd, vd, causal, p)
        m.mercury_sync_status()
        assert_close(out.cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref,
                     "R%d Rq%d runs%d" % (p.R, p.Rq, p.n_runs))


@pytest.mark.gpu
def test_tune_caches_and_rechecks(gpu):
    import oracle
    m = gpu
    B, Hq, Hkv, Sq, Skv, d, causal, R, shift = 1, 8, 1, 256, 32768, 128, False, 16, 1
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, d, seed=404)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o_ref, l_ref = oracle.attn(q, k, v, causal)
    m.mercury_tune_cache_clear()
    out, lse, best, hit = m.mercury_tune_schedule(qd, kd, vd, R, shift, causal, 0, 4)
    assert not hit and best.measured_us > 0 and best.R == R
    assert_close(out.cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, "tuned")
    out.zero_()
    out, lse, best2, hit = m.mercury_tune_schedule(qd, kd, vd, R, shift, causal, 0, 4, out=out, lse=lse)
    assert hit and (best2.R, best2.Rq, best2.n_runs) == (best.R, best.Rq, best.n_runs)
    assert_close(out.cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, "cached")
    # a tight budget is a different key and admits only the fused schedule
    io = io_bytes(B, Hq, Hkv, Sq, Skv, d)
    out, lse, best3, hit = m.mercury_tune_schedule(qd, kd, vd, R, shift, causal, io, 4)
    assert not hit and best3.n_runs == 1 and best3.hbm_bytes <= io
    assert_close(out.cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, "budget")
    m.mercury_tune_cache_clear()
    _, _, _, hit = m.mercury_tune_schedule(qd, kd, vd, R, shift, causal, 0, 4)
    assert not hit


@pytest.mark.gpu
def test_tune_recheck_drops_a_slow_entry(gpu, monkeypatch):
    """A cached schedule that misses its recorded time by more than the
    re-check factor is dropped and tuned again (factor 0: always)."""
    import oracle
    m = gpu
    B, Hq, Hkv, Sq, Skv, d, causal, R, shift = 1, 4, 2, 512, 4096, 128, True, 8, 4
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, d, seed=405)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    m.mercury_tune_cache_clear()
    _, _, _, hit = m.mercury_tune_schedule(qd, kd, vd, R, shift, causal, 0, 2)
    assert not hit
    _, _, _, hit = m.mercury_tune_schedule(qd, kd, vd, R, shift, causal, 0, 2)
    assert hit
    monkeypatch.setenv("MERCURY_TUNE_RECHECK", "0")
    out, lse, best, hit = m.mercury_tune_schedule(qd, kd, vd, R, shift, causal, 0, 2)
    assert not hit and best.measured_us > 0
    o_ref, l_ref = oracle.attn(q, k, v, causal)
    assert_close(out.cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, "re-tuned")
    m.mercury_tune_cache_clear()


@pytest.mark.gpu
def test_measured_profile_is_plausible_and_predicts(gpu):
    import torch
    m = gpu
    prof = m.mercury_measure_cost_profile()
    assert prof.measured == 1
    assert prof.n_sms == torch.cuda.get_device_properties(0).multi_processor_count
    assert 0.2 < prof.tile_us < 20 and 0 < prof.tile1_us <= prof.tile_us * 1.2
    assert 0 <= prof.item_us < 100 and 0 <= prof.launch_us < 200
    assert 500 < prof.merge_gbs < 20000 and 500 < prof.hbm_gbs < 20000
    # the estimate of a long causal GQA call (the bench shape) is within 30 % of
    # its measured time
    B, Hq, Hkv, Sq, Skv, d, causal, R, shift = 1, 32, 8, 32768, 32768, 128, True, 8, 1
    plans, _ = m.mercury_plan_schedules(B, Hq, Hkv, Sq, Skv, d, causal, R, shift, 0, prof, 1)
    q, k, v = (x.cuda() for x in make_qkv(B, Hq, Hkv, Sq, Skv, d, seed=9))
    out = torch.empty((B, Hq, Sq, d), device="cuda")
    lse = torch.empty((B, Hq, Sq), device="cuda")
    for _ in range(3):
        m.mercury_attn_run_schedule(q, k, v, causal, plans[0], out, lse)
    ts = []
    for _ in range(5):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        m.mercury_attn_run_schedule(q, k, v, causal, plans[0], out, lse)
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b) * 1e3)
    m.mercury_sync_status()
    measured = sorted(ts)[2]
    assert abs(plans[0].predicted_us - measured) <= 0.3 * measured, (plans[0].predicted_us, measured)
