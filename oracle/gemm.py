"""fp64 CPU oracle for the shifted-shard GEMM (test infrastructure only).

The pages' second operator family is the all-gather GEMM: every rank owns a
slice of A while all ranks need B, and instead of replicating B first, a rank
reads B's pieces from their owners in a rank-staggered order (Silicon &
Systems, "The hidden cost of synchronized operators"; "What Mercury finds that
templates miss", A100 all-gather GEMM).  Reading taken here: R virtual ranks;
rank i owns the row block A_i = A[i*M/R:(i+1)*M/R, :]; B is split into R
column shards B_s = B[:, s*N/R:(s+1)*N/R]; at step j rank i reads shard
s = order[i][j] (the shift primitive's (j+i)%J, or its nested / unshifted
forms, from this oracle's own table) and writes C[block i, shard s] =
A_i @ B_s.  The result is the plain product C = A @ B.

The matmul of each block is a library primitive (numpy, fp64) on the exactly
widened bf16 inputs; no blocking beyond the rank/shard split.
"""
from __future__ import annotations

import numpy as np

from . import _bf16_bits, shift_order


def _f64(x) -> np.ndarray:
    bits = _bf16_bits(x)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def gemm(a, b) -> np.ndarray:
    """C = A @ B in fp64; a [M, K], b [K, N] bf16."""
    return _f64(a) @ _f64(b)


def gemm_shifted(a, b, R: int, shift: int, return_visits: bool = False):
    """The shifted schedule: rank i, step j computes C[block i, shard order[i][j]]."""
    A, Bm = _f64(a), _f64(b)
    M, K = A.shape
    N = Bm.shape[1]
    if M % R or N % R:
        raise ValueError("R must divide M and N")
    Mr, Nr = M // R, N // R
    order = shift_order(R, shift)
    C = np.full((M, N), np.nan)
    visits = []
    for j in range(R):
        for i in range(R):
            s = int(order[i, j])
            C[i * Mr:(i + 1) * Mr, s * Nr:(s + 1) * Nr] = A[i * Mr:(i + 1) * Mr] @ Bm[:, s * Nr:(s + 1) * Nr]
            visits.append((i, j, s))
    return (C, visits) if return_visits else C
