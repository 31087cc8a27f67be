"""The shifted schedule across devices: virtual rank i on process (GPU) i.

On one GPU the R virtual ranks share HBM and "reading shard (i+j) mod R" is
a tile load from that shard's address.  Across devices the pages' form
applies: the KV buffer stays sharded over the devices' memory, every rank
consumes the shards in its own staggered order instead of all ranks taking
the same piece at the same time, and a piece moves when a consumer needs it
(Silicon & Systems, "The hidden cost of synchronized operators"; the shift
primitive's (j+i)%J access, Mercury-SOSP25 paper notes, 核心方法).  On a
two-level topology the order is nested so that most steps use the fast
inner links (Silicon & Systems, "What Mercury finds that templates miss").

This module is the host side of that form:

* ``exchange_plan(R, shift)`` -- for every step j >= 1 and rank i, the rank
  that sends i the shard it needs at step j and the rank i sends its
  step-(j-1) shard to.  A shard is passed on by whoever held it at the
  previous step, so the flat order becomes a ring (neighbour i+1 -> i) and
  the nested Ro x Ri order an inner ring inside each group with one hop
  across groups every Ri steps.  Every step is a bijection of ranks.  The
  unshifted order (every rank on shard j at step j) is the synchronous
  schedule: each step is a broadcast from the shard's owner.
* ``ShiftedKV`` -- rank i holds query block i and KV shard i.  At step j it
  runs the local attention patch on the shard in its current buffer while the
  shard of step j+1 arrives into the other buffer (point-to-point send and
  receive of the step's pairs, double-buffered), and folds the step's
  partial (O, LSE) into its running result with the log-sum-exp merge.
* ``ShiftedPartials`` -- the alternative that keeps every KV shard where it
  is and moves only results: with the (small) query side present on every
  rank, rank i computes the partial of every query block against its own
  shard, sends each partial to the block's owner in the shifted order, and
  each owner merges the partials of its block.

The exchange runs through ``torch.distributed`` point-to-point calls, so
the same code runs with the gloo backend on CPU tensors (how it is tested
here) and with NCCL on GPU tensors, where every remote shard lands in the
receiving GPU's own memory before a kernel reads it.  The local patch and the
merge are passed in: on GPUs they are this library's calls
(``cuda_patch`` / ``cuda_merge`` below), in CPU tests any implementation of
the same definition.  Causal masking across shards needs Sq == Skv (every
causal workload here): a shard before the query block is unmasked, the
diagonal shard is masked inside, a later shard contributes nothing.
"""
from __future__ import annotations

from typing import Callable, List, Optional, Sequence, Tuple

import numpy as np


def shift_table(R: int, shift: int) -> np.ndarray:
    """order[i][j] = shard that virtual rank i reads at step j (the encoding of
    mercury_plan_shift: 0 unshifted, 1 flat (i + j) mod R, k >= 2 nested with
    inner size k).  Host arithmetic only; the C planner computes the same
    table, which the tests compare."""
    if R < 1 or shift < 0 or (shift >= 2 and R % shift != 0):
        raise ValueError("invalid (R, shift) = (%d, %d)" % (R, shift))
    order = np.empty((R, R), dtype=np.int64)
    for i in range(R):
        for j in range(R):
            if shift == 0:
                order[i, j] = j
            elif shift == 1:
                order[i, j] = (i + j) % R
            else:
                Ri, Ro = shift, R // shift
                order[i, j] = ((i // Ri + j // Ri) % Ro) * Ri + (i % Ri + j % Ri) % Ri
    return order


def exchange_plan(R: int, shift: int) -> List[Optional[List[Tuple[int, int]]]]:
    """Point-to-point pairs of the pass-along exchange.

    plan[0] is None (every rank starts with its own shard, order[i][0] = i
    for the shifted orders).  For j >= 1, plan[j][i] = (src, dst): rank i
    receives the shard it reads at step j from `src`, which held it at step
    j-1, and sends the shard it held at step j-1 to `dst`, which reads it at
    step j.  For the unshifted order (shift 0) there is no pass-along: the
    plan is None at every step and each step is a broadcast from rank j."""
    order = shift_table(R, shift)
    if shift == 0:
        return [None] * R
    plan: List[Optional[List[Tuple[int, int]]]] = [None]
    for j in range(1, R):
        holder_prev = {int(order[r, j - 1]): r for r in range(R)}   # shard -> rank at step j-1
        reader_now = {int(order[r, j]): r for r in range(R)}        # shard -> rank at step j
        plan.append([(holder_prev[int(order[i, j])], reader_now[int(order[i, j - 1])]) for i in range(R)])
    return plan


def partial_plan(R: int, shift: int) -> List[List[Tuple[int, int]]]:
    """Pairs of the partial-exchange form: at step j rank i computes the
    partial of query block p (the rank that reads shard i at step j, i.e.
    order[p][j] = i) against its own shard i and sends it to p; it receives
    from the rank order[i][j] the partial of its own block against that
    rank's shard.  plan[j][i] = (src, dst) = (order[i][j], p).  Shifted orders
    only (shift >= 1): under the unshifted order every rank reads the same
    shard at a step, so its owner would have to serve all blocks at once."""
    if shift == 0:
        raise ValueError("the partial exchange needs a shifted order (shift >= 1)")
    order = shift_table(R, shift)
    plan = []
    for j in range(R):
        reader = {int(order[r, j]): r for r in range(R)}
        plan.append([(int(order[i, j]), reader[i]) for i in range(R)])
    return plan


def causal_relation(block: int, shard: int) -> str:
    """How query block `block` sees KV shard `shard` under the causal mask
    when Sq == Skv and both are cut into R equal pieces: 'full' (every key
    allowed), 'diagonal' (masked inside the shard) or 'none'."""
    if shard < block:
        return "full"
    if shard == block:
        return "diagonal"
    return "none"


Patch = Callable[..., Tuple[object, object]]
Merge = Callable[[Tuple[object, object], Tuple[object, object]], Tuple[object, object]]


class ShiftedKV:
    """KV shards travel; each rank keeps its query block and its result.

    patch(q, k, v, relation) -> (o, lse): attention of the query block over
    one shard with relation in {'full', 'diagonal'} (non-causal calls always
    pass 'full'); merge((o1, l1), (o2, l2)) -> (o, l): the log-sum-exp
    merge of two partials.  Both run on whatever device the tensors live on.
    Messages are sent as bytes, so any dtype travels (gloo has no bf16).
    """

    def __init__(self, R: int, shift: int, causal: bool, rank: int, group=None, record_checksums: bool = False):
        import torch.distributed as dist
        self.dist = dist
        self.R, self.shift, self.causal, self.rank, self.group = R, shift, bool(causal), rank, group
        self.order = shift_table(R, shift)
        self.plan = exchange_plan(R, shift)
        if dist.get_world_size(group) != R:
            raise ValueError("the process group must have R = %d ranks" % R)
        self.received: List[int] = []      # shard index used at each step
        # Sum of each step's shard (record_checksums=True, for checks only: it
        # reads the shard back to the host every step, which serialises the
        # exchange with the compute).
        self.record_checksums = record_checksums
        self.checksums: List[float] = []

    def _global(self, r: int) -> int:
        return r if self.group is None else self.dist.get_global_rank(self.group, r)

    def _start(self, j: int, own, cur, nxt):
        """Start bringing the shard of step j into `nxt`: the pass-along pair of
        the step, or, for the unshifted order, a broadcast from its owner j."""
        dist = self.dist
        if self.shift == 0:
            if self.rank == j:
                nxt.copy_(own)
            return [dist.broadcast(nxt.view(-1).view(_u8()), src=self._global(j), group=self.group,
                                   async_op=True)]
        src, dst = self.plan[j][self.rank]
        ops = [dist.P2POp(dist.isend, cur.view(-1).view(_u8()), self._global(dst), self.group),
               dist.P2POp(dist.irecv, nxt.view(-1).view(_u8()), self._global(src), self.group)]
        return dist.batch_isend_irecv(ops)

    def run(self, q, k_shard, v_shard, patch: Patch, merge: Merge):
        import torch
        own = torch.stack([k_shard, v_shard]).contiguous()   # one message per step
        bufs = [torch.empty_like(own), torch.empty_like(own)]
        if self.shift == 0:
            for w in self._start(0, own, None, bufs[0]):
                w.wait()
        else:
            bufs[0].copy_(own)                               # order[i][0] = i
        acc = None
        self.received, self.checksums = [], []
        for j in range(self.R):
            cur, nxt = bufs[j % 2], bufs[(j + 1) % 2]
            # the next step's shard moves while this step's patch runs
            works = self._start(j + 1, own, cur, nxt) if j + 1 < self.R else []
            s = int(self.order[self.rank, j])
            self.received.append(s)
            if self.record_checksums:
                self.checksums.append(float(cur.double().sum()))
            rel = causal_relation(self.rank, s) if self.causal else "full"
            if rel != "none":
                part = patch(q, cur[0], cur[1], rel)
                acc = part if acc is None else merge(acc, part)
            for w in works:
                w.wait()
        return acc


def _u8():
    import torch
    return torch.uint8


class ShiftedPartials:
    """KV shards stay; partial results travel.  Every rank holds the whole
    (short) query side q_all [B, Hq, Sq, d] and its KV shard; it returns the
    merged result of its own query block."""

    def __init__(self, R: int, shift: int, causal: bool, rank: int, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.R, self.shift, self.causal, self.rank, self.group = R, shift, bool(causal), rank, group
        self.order = shift_table(R, shift)
        self.plan = partial_plan(R, shift)
        if dist.get_world_size(group) != R:
            raise ValueError("the process group must have R = %d ranks" % R)

    def _global(self, r: int) -> int:
        return r if self.group is None else self.dist.get_global_rank(self.group, r)

    def run(self, q_all, k_shard, v_shard, patch: Patch, merge: Merge, empty_partial):
        """empty_partial(q_block) -> (o, lse) of a block that sees no key (O = 0,
        LSE = -inf): sent when a causal block lies before this rank's shard."""
        import torch
        dist = self.dist
        Sq = q_all.shape[2]
        Bq = Sq // self.R
        acc = None
        self.sources: List[int] = []
        for j in range(self.R):
            src, dst = self.plan[j][self.rank]
            qb = q_all[:, :, dst * Bq:(dst + 1) * Bq].contiguous()
            rel = causal_relation(dst, self.rank) if self.causal else "full"
            o, l = patch(qb, k_shard, v_shard, rel) if rel != "none" else empty_partial(qb)
            if src == self.rank:
                # step 0 of a shifted order: the block's own shard, nothing moves
                assert dst == self.rank
                part = (o, l)
            else:
                send = torch.cat([o.reshape(-1), l.reshape(-1)]).contiguous()
                recv = torch.empty_like(send)
                works = dist.batch_isend_irecv([
                    dist.P2POp(dist.isend, send.view(_u8()), self._global(dst), self.group),
                    dist.P2POp(dist.irecv, recv.view(_u8()), self._global(src), self.group)])
                for w in works:
                    w.wait()
                n_o = o.numel()
                part = (recv[:n_o].view_as(o), recv[n_o:].view_as(l))
            self.sources.append(src)
            acc = part if acc is None else merge(acc, part)
        return acc


# ------------------------------------------------------------ GPU patch

def cuda_patch(q, k, v, relation: str):
    """The local attention patch on a GPU: this library's fused call on one
    (query block, KV shard) pair, one virtual rank, fp32 O and LSE."""
    from . import mercury as m
    return m.mercury_attn_sharded(q, k, v, 1, 1, relation == "diagonal")


def cuda_merge(a, b):
    """Log-sum-exp merge of two partials with this library's merge kernel."""
    import torch
    from . import mercury as m
    o = torch.stack([a[0], b[0]])
    l = torch.stack([a[1], b[1]])
    return m.mercury_lse_merge(o, l)


def cuda_empty_partial(qb):
    import torch
    o = torch.zeros(qb.shape, dtype=torch.float32, device=qb.device)
    l = torch.full(qb.shape[:-1], float("-inf"), dtype=torch.float32, device=qb.device)
    return o, l
