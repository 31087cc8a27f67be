"""Pins of the shifted-shard GEMM oracle: identity and one-hot closed forms,
a triple-loop brute force, and the shifted schedule visiting every (rank,
shard) block exactly once in the shift table's order."""
import numpy as np
import pytest
import torch

from oracle import gemm as og
from tests.conftest import load_golden_table


def bf16(x):
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def rnd(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(torch.bfloat16)


def test_identity_gives_b():
    b = rnd((64, 48), 1)
    c = og.gemm(bf16(np.eye(64)), b)
    np.testing.assert_array_equal(c, b.double().numpy())


def test_one_hot_rows_select_b_rows():
    b = rnd((32, 40), 2)
    a = np.zeros((5, 32), np.float32)
    picks = [3, 0, 31, 17, 3]
    for r, k in enumerate(picks):
        a[r, k] = 2.0
    c = og.gemm(bf16(a), b)
    np.testing.assert_array_equal(c, 2.0 * b.double().numpy()[picks])


@pytest.mark.parametrize("M,K,N", [(1, 1, 1), (3, 5, 2), (8, 16, 12)])
def test_brute_force_triple_loop(M, K, N):
    a, b = rnd((M, K), M + K), rnd((K, N), N)
    c = og.gemm(a, b)
    A, B = a.double().numpy(), b.double().numpy()
    for i in range(M):
        for j in range(N):
            ref = 0.0
            for k in range(K):
                ref += A[i, k] * B[k, j]
            assert abs(c[i, j] - ref) < 1e-12


@pytest.mark.parametrize("R,shift", [(1, 1), (2, 1), (4, 0), (4, 1), (8, 1), (8, 4), (8, 2)])
def test_shifted_schedule_equals_plain(R, shift):
    a, b = rnd((64, 24), R), rnd((24, 32), shift + 7)
    c, visits = og.gemm_shifted(a, b, R, shift, return_visits=True)
    np.testing.assert_allclose(c, og.gemm(a, b), atol=1e-12, rtol=0)
    assert sorted((i, s) for i, _, s in visits) == [(i, s) for i in range(R) for s in range(R)]


@pytest.mark.parametrize("R,shift,name", [(4, 1, "shift_R4_flat.txt"), (8, 4, "shift_R8_nested_2x4.txt")])
def test_shifted_visit_order_follows_table(R, shift, name):
    a, b = rnd((8 * R, 8), 1), rnd((8, 8 * R), 2)
    _, visits = og.gemm_shifted(a, b, R, shift, return_visits=True)
    table = load_golden_table(name)
    for i, j, s in visits:
        assert table[i][j] == s
