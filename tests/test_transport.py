"""The shifted schedule across processes (virtual rank i on process i), on CPU
gloo ranks with the fp64 oracle as the local patch.

Host logic first: the exchange plan of every step is a bijection, passing
shards along it makes every rank hold exactly shard order[i][j] at step j,
the nested order keeps its inner steps inside a group, and the module's
shift table equals the C planner's and the oracle's.  Then 2, 4 and 8 gloo
ranks run both forms -- KV shards travel (ShiftedKV) and only partial
results travel (ShiftedPartials) -- for flat, nested and unshifted orders,
causal and not: each rank must see the shards in its shifted order, with the
bytes of the true shard, and its block of the result must equal plain
attention (the oracle on the whole input) to fp64 rounding.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from long_context_sharded_gb300 import transport as tp


@pytest.mark.parametrize("R", [1, 2, 3, 4, 6, 8, 16])
def test_shift_table_matches_planner_and_oracle(R):
    import oracle
    from long_context_sharded_gb300 import build
    build.build()
    from long_context_sharded_gb300 import mercury as m
    for shift in [0, 1] + [k for k in range(2, R + 1) if R % k == 0]:
        t = tp.shift_table(R, shift)
        assert (t == m.mercury_plan_shift(R, shift)).all()
        assert (t == oracle.shift_order(R, shift)).all()


@pytest.mark.parametrize("R,shift", [(2, 1), (4, 1), (8, 1), (5, 1), (4, 2), (8, 4), (8, 2), (16, 4), (12, 3)])
def test_exchange_plan_passes_every_shard_to_its_reader(R, shift):
    order = tp.shift_table(R, shift)
    plan = tp.exchange_plan(R, shift)
    assert plan[0] is None and len(plan) == R
    held = [int(order[i, 0]) for i in range(R)]
    assert held == list(range(R))                     # rank i starts with its own shard
    for j in range(1, R):
        pairs = plan[j]
        srcs = sorted(p[0] for p in pairs)
        dsts = sorted(p[1] for p in pairs)
        assert srcs == list(range(R)) and dsts == list(range(R))   # bijections
        for i, (src, dst) in enumerate(pairs):
            assert pairs[dst][0] == i                 # my receiver receives from me
            assert pairs[src][1] == i                 # my sender sends to me
        held = [held[pairs[i][0]] for i in range(R)]
        assert held == [int(order[i, j]) for i in range(R)]


def test_flat_order_is_a_ring():
    R = 8
    for j, pairs in enumerate(tp.exchange_plan(R, 1)[1:], start=1):
        assert pairs == [((i + 1) % R, (i - 1) % R) for i in range(R)]


@pytest.mark.parametrize("R,Ri", [(8, 4), (8, 2), (16, 4)])
def test_nested_order_crosses_groups_only_at_outer_steps(R, Ri):
    """Inner steps pass shards inside a group of Ri ranks; only every Ri-th
    step crosses to another group (the hierarchical 2 x 4 / 4 x 2 form)."""
    plan = tp.exchange_plan(R, Ri)
    for j in range(1, R):
        crosses = [src // Ri != i // Ri for i, (src, _) in enumerate(plan[j])]
        if j % Ri:
            assert not any(crosses), j
        else:
            assert all(crosses), j
    flat = tp.exchange_plan(R, 1)
    flat_cross = sum(src // Ri != i // Ri for j in range(1, R) for i, (src, _) in enumerate(flat[j]))
    nested_cross = sum(src // Ri != i // Ri for j in range(1, R) for i, (src, _) in enumerate(plan[j]))
    assert nested_cross < flat_cross


@pytest.mark.parametrize("R,shift", [(4, 1), (8, 4), (6, 3), (8, 2)])
def test_partial_plan_is_a_bijection_per_step(R, shift):
    order = tp.shift_table(R, shift)
    plan = tp.partial_plan(R, shift)
    for j in range(R):
        assert sorted(p[0] for p in plan[j]) == list(range(R))
        assert sorted(p[1] for p in plan[j]) == list(range(R))
        for i, (src, dst) in enumerate(plan[j]):
            assert order[i, j] == src and order[dst, j] == i


def test_partial_plan_rejects_the_unshifted_order():
    with pytest.raises(ValueError):
        tp.partial_plan(4, 0)


def test_causal_relation():
    assert tp.causal_relation(3, 1) == "full"
    assert tp.causal_relation(3, 3) == "diagonal"
    assert tp.causal_relation(3, 4) == "none"


# ------------------------------------------------------------ gloo ranks

def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _oracle_patch(q, k, v, relation):
    import oracle
    o, l = oracle.attn(q, k, v, relation == "diagonal")
    return torch.from_numpy(np.ascontiguousarray(o)), torch.from_numpy(np.ascontiguousarray(l))


def _oracle_merge(a, b):
    import oracle
    shape_o, shape_l, d = a[0].shape, a[1].shape, a[0].shape[-1]
    o, l = oracle.lse_merge(np.stack([a[0].numpy().reshape(-1, d), b[0].numpy().reshape(-1, d)]),
                            np.stack([a[1].numpy().reshape(-1), b[1].numpy().reshape(-1)]))
    return (torch.from_numpy(np.ascontiguousarray(o)).view(shape_o),
            torch.from_numpy(np.ascontiguousarray(l)).view(shape_l))


def _empty_partial(qb):
    return (torch.zeros(qb.shape, dtype=torch.float64),
            torch.full(qb.shape[:-1], float("-inf"), dtype=torch.float64))


def _worker(rank, world, port, cfg, form, q_out):
    import torch.distributed as dist
    from long_context_sharded_gb300.inputs import make_qkv
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        B, Hq, Hkv, S, d, shift, causal = cfg
        R = world
        q, k, v = make_qkv(B, Hq, Hkv, S, S, d, seed=sum(cfg[:5]) + shift)
        Bq = S // R
        qi = q[:, :, rank * Bq:(rank + 1) * Bq].contiguous()
        ks = k[:, :, rank * Bq:(rank + 1) * Bq].contiguous()
        vs = v[:, :, rank * Bq:(rank + 1) * Bq].contiguous()
        if form == "kv":
            ex = tp.ShiftedKV(R, shift, causal, rank, record_checksums=True)
            o, l = ex.run(qi, ks, vs, _oracle_patch, _oracle_merge)
            true_sums = [float(torch.stack([k[:, :, s * Bq:(s + 1) * Bq], v[:, :, s * Bq:(s + 1) * Bq]])
                               .double().sum()) for s in ex.received]
            info = {"received": ex.received, "sums_ok": np.allclose(ex.checksums, true_sums, rtol=0, atol=0)}
        else:
            ex = tp.ShiftedPartials(R, shift, causal, rank)
            o, l = ex.run(q, ks, vs, _oracle_patch, _oracle_merge, _empty_partial)
            info = {"received": ex.sources, "sums_ok": True}
        q_out.put((rank, o.numpy(), l.numpy(), info))
    finally:
        dist.destroy_process_group()


CASES = [
    # (world, (B, Hq, Hkv, S, d, shift, causal), form)
    (2, (1, 2, 1, 64, 64, 1, True), "kv"),
    (2, (1, 2, 2, 64, 64, 1, False), "partial"),
    (4, (1, 4, 2, 128, 64, 1, True), "kv"),
    (4, (1, 2, 1, 128, 64, 2, True), "kv"),          # nested 2 x 2
    (4, (1, 2, 2, 128, 64, 0, False), "kv"),         # unshifted: broadcasts from the owner
    (4, (2, 2, 1, 64, 64, 1, True), "partial"),
    (8, (1, 4, 1, 256, 64, 4, True), "kv"),          # nested 2 x 4
    (8, (1, 2, 2, 128, 64, 4, False), "partial"),
]


@pytest.mark.parametrize("world,cfg,form", CASES, ids=lambda x: str(x).replace(" ", ""))
def test_ranks_compute_plain_attention(world, cfg, form):
    import oracle
    from long_context_sharded_gb300.inputs import make_qkv
    oracle.build()
    ctx = mp.get_context("spawn")
    q_out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, cfg, form, q_out)) for r in range(world)]
    for p in procs:
        p.start()
    res = []
    import queue
    import time
    t0 = time.time()
    while len(res) < world:
        try:
            res.append(q_out.get(timeout=1))
        except queue.Empty:
            dead = [p.exitcode for p in procs if p.exitcode not in (None, 0)]
            if dead or time.time() - t0 > 300:
                for p in procs:
                    if p.is_alive():
                        p.kill()
                pytest.fail("a rank failed (exit codes %s) or the ranks ran out of time" % dead)
    res.sort(key=lambda x: x[0])
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    B, Hq, Hkv, S, d, shift, causal = cfg
    q, k, v = make_qkv(B, Hq, Hkv, S, S, d, seed=sum(cfg[:5]) + shift)
    o_ref, l_ref = oracle.attn(q, k, v, causal)
    order = tp.shift_table(world, shift)
    Bq = S // world
    for rank, o, l, info in res:
        if form == "kv":
            assert info["received"] == [int(s) for s in order[rank]]
        else:
            assert info["received"] == [int(s) for s in order[rank]]
        assert info["sums_ok"]
        np.testing.assert_allclose(o, o_ref[:, :, rank * Bq:(rank + 1) * Bq], rtol=0, atol=1e-10)
        np.testing.assert_allclose(l, l_ref[:, :, rank * Bq:(rank + 1) * Bq], rtol=0, atol=1e-10)


# ------------------------------------------------------------ GPU patch

def _emulate_ranks(R, shift, causal, q, k, v, patch, merge):
    """All R ranks of ShiftedKV in one process: shards are passed along the
    exchange plan with plain copies (what the point-to-point calls do between
    processes), each rank runs the patch on the shard it holds."""
    order = tp.shift_table(R, shift)
    plan = tp.exchange_plan(R, shift)
    n = q.shape[2] // R
    blk = lambda t, i: t[:, :, i * n:(i + 1) * n].contiguous()  # noqa: E731
    held = [torch.stack([blk(k, i), blk(v, i)]) for i in range(R)]
    if shift == 0:
        held = [torch.stack([blk(k, 0), blk(v, 0)]) for _ in range(R)]
    acc = [None] * R
    for j in range(R):
        if j > 0:
            if shift == 0:
                held = [torch.stack([blk(k, j), blk(v, j)]) for _ in range(R)]
            else:
                held = [held[plan[j][i][0]].clone() for i in range(R)]
        for i in range(R):
            s = int(order[i, j])
            assert torch.equal(held[i][0], blk(k, s))
            rel = tp.causal_relation(i, s) if causal else "full"
            if rel == "none":
                continue
            part = patch(blk(q, i), held[i][0], held[i][1], rel)
            acc[i] = part if acc[i] is None else merge(acc[i], part)
    return acc


@pytest.mark.gpu
@pytest.mark.parametrize("R,shift,causal", [(2, 1, True), (4, 1, False), (8, 4, True), (4, 2, True), (4, 0, False)])
def test_gpu_patch_and_merge_through_the_exchange(R, shift, causal):
    """The GPU pieces of the multi-GPU form -- this library's fused call as
    the per-(block, shard) patch and its merge kernel -- fed shard by shard
    in the exchange plan's order, give plain attention for every block."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import oracle
    from long_context_sharded_gb300 import build
    from long_context_sharded_gb300.inputs import make_qkv
    build.build()
    B, Hq, Hkv, S, d = 1, 8, 2, 1024, 128
    q, k, v = make_qkv(B, Hq, Hkv, S, S, d, seed=R * 10 + shift)
    acc = _emulate_ranks(R, shift, causal, q.cuda(), k.cuda(), v.cuda(), tp.cuda_patch, tp.cuda_merge)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.attn(q, k, v, causal)
    n = S // R
    for i, (o, l) in enumerate(acc):
        err = np.abs(o.cpu().double().numpy() - o_ref[:, :, i * n:(i + 1) * n])
        assert err.max() <= 2e-2 and err.mean() <= 2e-3, (i, err.max(), err.mean())
        assert np.abs(l.cpu().double().numpy() - l_ref[:, :, i * n:(i + 1) * n]).max() <= 1e-3
