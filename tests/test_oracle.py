"""Pins of the fp64 CPU oracle against what the pages and the mathematics fix.

The pages print no worked attention example, so every pin here is a closed
form, an invariant, a hand-written table or an independent brute force:
  * hand-written shift tables (the (j+i)%J rule, and the nested reading),
  * Q = 0 gives the mean of the allowed V rows and LSE = ln(#allowed),
  * a dominant one-hot score selects its V row (closed-form LSE),
  * constant V passes through unchanged,
  * causal row 0 sees only key 0; causal and non-causal agree on the last row,
  * GQA equals MHA with K/V repeated per group,
  * every shift order and every R gives the unsharded result,
  * the merge is permutation invariant, and two equal-LSE partials average,
  * numpy brute force and torch fp64 SDPA (a library call) agree on tiny shapes.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from tests.conftest import load_golden_table


def bf16(x):
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.contiguous()


def rand_qkv(B, Hq, Hkv, Sq, Skv, d, seed, scale=1.0):
    from long_context_sharded_gb300.inputs import make_qkv
    return make_qkv(B, Hq, Hkv, Sq, Skv, d, seed=seed, scale=scale)


def f64(t):
    return t.to(torch.float64).numpy()


# ---------------------------------------------------------------- shift table

@pytest.mark.parametrize("R,shift,name", [(4, 1, "shift_R4_flat.txt"),
                                          (4, 0, "shift_R4_unshifted.txt"),
                                          (8, 4, "shift_R8_nested_2x4.txt")])
def test_shift_table_golden(R, shift, name):
    assert oracle.shift_order(R, shift).tolist() == load_golden_table(name)


@pytest.mark.parametrize("R", [1, 2, 3, 4, 6, 8, 12, 16, 64])
def test_shift_latin_square(R):
    shifts = [1] + [k for k in range(2, R + 1) if R % k == 0]
    for shift in shifts:
        t = oracle.shift_order(R, shift)
        for i in range(R):
            assert sorted(t[i].tolist()) == list(range(R))      # each rank sees each shard once
            assert sorted(t[:, i].tolist()) == list(range(R))   # each step is a bijection
        assert t[:, 0].tolist() == list(range(R))               # step 0: own shard


@pytest.mark.parametrize("R", [2, 4, 8, 16])
def test_nested_with_one_outer_group_is_flat(R):
    assert (oracle.shift_order(R, R) == oracle.shift_order(R, 1)).all()


def test_shift_invalid():
    with pytest.raises(ValueError):
        oracle.shift_order(8, 3)
    with pytest.raises(ValueError):
        oracle.shift_order(0, 1)


# ------------------------------------------------------------- closed forms

@pytest.mark.parametrize("causal,Sq,Skv", [(False, 16, 16), (True, 16, 16),
                                           (True, 8, 24), (False, 5, 37)])
def test_q_zero_gives_mean_of_allowed_v(causal, Sq, Skv):
    d = 64
    _, k, v = rand_qkv(1, 2, 1, Sq, Skv, d, seed=11)
    q = torch.zeros(1, 2, Sq, d, dtype=torch.bfloat16)
    out, lse = oracle.attn(q, k, v, causal)
    vv = f64(v)[0, 0]
    for h in range(2):
        for qi in range(Sq):
            n = (qi + (Skv - Sq) + 1) if causal else Skv
            np.testing.assert_allclose(out[0, h, qi], vv[:n].mean(axis=0), rtol=0, atol=1e-13)
            assert abs(lse[0, h, qi] - math.log(n)) < 1e-13


@pytest.mark.parametrize("d,alpha", [(64, 16.0), (128, 24.0)])
def test_one_hot_dominant_selects_row(d, alpha):
    S = 32
    kstar = 13
    q = np.zeros((1, 1, S, d), np.float32)
    q[..., 0] = alpha
    k = np.zeros((1, 1, S, d), np.float32)
    rng = np.random.default_rng(3)
    k[0, 0, :, 1:] = np.round(rng.standard_normal((S, d - 1)) * 4) / 64.0   # small, bf16-exact
    k[0, 0, :, 0] = 0.0
    k[0, 0, kstar, :] = 0.0
    k[0, 0, kstar, 0] = alpha
    v = np.round(rng.standard_normal((1, 1, S, d)) * 8) / 8.0
    out, lse = oracle.attn(bf16(q), bf16(k), bf16(v), causal=False)
    gap = alpha * alpha / math.sqrt(d)            # score of k*, others score exactly 0
    n = S
    expect_lse = gap + math.log1p((n - 1) * math.exp(-gap))
    bound = n * math.exp(-gap) * np.abs(v).max() * 2
    for qi in range(S):
        np.testing.assert_allclose(out[0, 0, qi], v[0, 0, kstar], atol=bound, rtol=0)
        assert abs(lse[0, 0, qi] - expect_lse) < 1e-12


def test_constant_v_passes_through():
    q, k, _ = rand_qkv(2, 4, 2, 24, 24, 64, seed=5)
    c = np.linspace(-2, 2, 64).astype(np.float32)
    c = np.round(c * 16) / 16
    v = np.broadcast_to(c, (2, 2, 24, 64)).copy()
    for causal in (False, True):
        out, _ = oracle.attn(q, k, bf16(v), causal)
        np.testing.assert_allclose(out, np.broadcast_to(c, out.shape), atol=1e-13, rtol=0)


def test_causal_row0_sees_only_key0():
    d = 64
    q = np.zeros((1, 1, 8, d), np.float32)
    k = np.zeros((1, 1, 8, d), np.float32)
    q[0, 0, 0, 0], q[0, 0, 0, 1] = 1.5, -2.0
    k[0, 0, 0, 0], k[0, 0, 0, 1] = 3.0, 0.25
    k[0, 0, 1:, :] = 9.0                         # huge scores, but masked for row 0
    _, _, v = rand_qkv(1, 1, 1, 8, 8, d, seed=9)
    out, lse = oracle.attn(bf16(q), bf16(k), v, causal=True)
    np.testing.assert_allclose(out[0, 0, 0], f64(v)[0, 0, 0], atol=1e-14, rtol=0)
    assert abs(lse[0, 0, 0] - (1.5 * 3.0 - 2.0 * 0.25) / math.sqrt(d)) < 1e-14


def test_causal_last_row_equals_noncausal():
    q, k, v = rand_qkv(1, 2, 2, 20, 20, 64, seed=4)
    oc, lc = oracle.attn(q, k, v, True)
    on, ln = oracle.attn(q, k, v, False)
    np.testing.assert_allclose(oc[:, :, -1], on[:, :, -1], atol=1e-14, rtol=0)
    np.testing.assert_allclose(lc[:, :, -1], ln[:, :, -1], atol=1e-14, rtol=0)
    assert np.abs(oc[:, :, 0] - on[:, :, 0]).max() > 1e-3   # mask actually bites


def test_gqa_equals_repeated_mha():
    q, k, v = rand_qkv(2, 8, 2, 16, 16, 64, seed=8)
    for causal in (False, True):
        og, lg = oracle.attn(q, k, v, causal)
        om, lm = oracle.attn(q, k.repeat_interleave(4, dim=1), v.repeat_interleave(4, dim=1), causal)
        np.testing.assert_array_equal(og, om)
        np.testing.assert_array_equal(lg, lm)
    # the mapping is h // G (consecutive heads share a kv head), not h % Hkv
    o_wrong, _ = oracle.attn(q, k.repeat(1, 4, 1, 1), v.repeat(1, 4, 1, 1), False)
    og, _ = oracle.attn(q, k, v, False)
    assert np.abs(o_wrong - og).max() > 1e-3


# ------------------------------------------------------------- brute force

@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,d", [(1, 1, 1, 1, 1, 4), (2, 4, 2, 7, 7, 8),
                                               (1, 2, 1, 5, 16, 8), (2, 2, 2, 16, 16, 64),
                                               (1, 4, 1, 3, 9, 4)])
@pytest.mark.parametrize("causal", [False, True])
def test_brute_force_tiny(B, Hq, Hkv, Sq, Skv, d, causal):
    q, k, v = rand_qkv(B, Hq, Hkv, Sq, Skv, d, seed=B * 100 + Sq + d)
    out, lse = oracle.attn(q, k, v, causal)
    ob, lb = brute.attention(f64(q), f64(k), f64(v), causal)
    np.testing.assert_allclose(out, ob, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse, lb, atol=1e-12, rtol=0)
    # a library routine as a third, independent check
    G = Hq // Hkv
    qt, kt, vt = (x.to(torch.float64) for x in (q, k, v))
    kt, vt = kt.repeat_interleave(G, dim=1), vt.repeat_interleave(G, dim=1)
    mask = None
    if causal:
        qi = torch.arange(Sq)[:, None]
        ki = torch.arange(Skv)[None, :]
        mask = ki <= qi + (Skv - Sq)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask)
    np.testing.assert_allclose(out, ref.numpy(), atol=1e-12, rtol=0)


def test_brute_bf16_widening_exact():
    vals = np.array([0.0, -0.0, 1.0, -2.5, 3.140625, 1e-30, 6.5e4, -1e30], np.float32)
    t = bf16(vals)
    bits = t.view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(brute.bf16_bits_to_f64(bits), t.to(torch.float64).numpy())


# ------------------------------------------------------ sharding and merging

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("R,shift", [(1, 1), (2, 1), (4, 0), (4, 1), (4, 2), (8, 1), (8, 4), (8, 2), (16, 1)])
def test_sharded_equals_unsharded(R, shift, causal):
    q, k, v = rand_qkv(1, 4, 2, 32, 32, 64, seed=R * 10 + shift)
    o0, l0 = oracle.attn(q, k, v, causal)
    o1, l1 = oracle.attn_sharded(q, k, v, R, shift, causal)
    np.testing.assert_allclose(o1, o0, atol=1e-12, rtol=0)
    np.testing.assert_allclose(l1, l0, atol=1e-12, rtol=0)


def test_sharded_uneven_lengths_causal():
    q, k, v = rand_qkv(1, 2, 1, 16, 48, 64, seed=77)
    o0, l0 = oracle.attn(q, k, v, True)
    for shift in (0, 1, 2):
        o1, l1 = oracle.attn_sharded(q, k, v, 4, shift, True)
        np.testing.assert_allclose(o1, o0, atol=1e-12, rtol=0)
        np.testing.assert_allclose(l1, l0, atol=1e-12, rtol=0)


def test_partials_follow_shift_order_and_mask():
    R = 4
    q, k, v = rand_qkv(1, 1, 1, 16, 16, 64, seed=21)
    op, lp = oracle.attn_partial(q, k, v, R, 1, causal=True)
    Bq = 4
    for qi in range(16):
        i = qi // Bq
        for j in range(R):
            s = (i + j) % R
            if s > i:      # shard entirely in the future of this rank: masked
                assert lp[j, 0, 0, qi] == -np.inf
                assert not op[j, 0, 0, qi].any()
            else:
                # slot j equals plain attention restricted to shard s
                hi = min(qi, (s + 1) * Bq - 1)
                kk, vv = k[:, :, s * Bq:hi + 1], v[:, :, s * Bq:hi + 1]
                o_s, l_s = oracle.attn(q[:, :, qi:qi + 1], kk, vv, False)
                np.testing.assert_allclose(op[j, 0, 0, qi], o_s[0, 0, 0], atol=1e-13, rtol=0)
                assert abs(lp[j, 0, 0, qi] - l_s[0, 0, 0]) < 1e-13


def test_merge_permutation_invariant():
    R = 8
    q, k, v = rand_qkv(1, 2, 2, 32, 32, 64, seed=31)
    op, lp = oracle.attn_partial(q, k, v, R, 1, causal=True)
    o0, l0 = oracle.attn(q, k, v, True)
    rows = 2 * 32
    op = op.reshape(R, rows, 64)
    lp = lp.reshape(R, rows)
    rng = np.random.default_rng(5)
    for _ in range(4):
        perm = rng.permutation(R)
        om, lm = oracle.lse_merge(op[perm], lp[perm])
        np.testing.assert_allclose(om, o0.reshape(rows, 64), atol=1e-12, rtol=0)
        np.testing.assert_allclose(lm, l0.reshape(rows), atol=1e-12, rtol=0)


def test_merge_two_equal_lse_partials_average():
    rng = np.random.default_rng(1)
    a = rng.standard_normal((5, 16))
    b = rng.standard_normal((5, 16))
    lse = rng.standard_normal(5) * 3
    om, lm = oracle.lse_merge(np.stack([a, b]), np.stack([lse, lse]))
    np.testing.assert_allclose(om, (a + b) / 2, atol=1e-15, rtol=0)
    np.testing.assert_allclose(lm, lse + math.log(2), atol=1e-14, rtol=0)


def test_merge_weights_closed_form():
    # weights exp(l_j - L) with L = ln(e^1 + e^2 + e^3)
    o = np.array([[[1.0, 0.0]], [[0.0, 1.0]], [[2.0, 2.0]]])
    l = np.array([[1.0], [2.0], [3.0]])
    om, lm = oracle.lse_merge(o, l)
    L = math.log(math.e + math.e ** 2 + math.e ** 3)
    w = [math.exp(1 - L), math.exp(2 - L), math.exp(3 - L)]
    assert abs(lm[0] - L) < 1e-14
    np.testing.assert_allclose(om[0], [w[0] + 2 * w[2], w[1] + 2 * w[2]], atol=1e-15, rtol=0)


def test_merge_masked_parts():
    o = np.zeros((3, 2, 4))
    o[1, 0] = [1, 2, 3, 4]
    l = np.full((3, 2), -np.inf)
    l[1, 0] = 0.7
    om, lm = oracle.lse_merge(o, l)
    np.testing.assert_array_equal(om[0], [1, 2, 3, 4])
    assert lm[0] == 0.7
    assert not om[1].any() and lm[1] == -np.inf
    assert not np.isnan(om).any()


def test_sampled_rows_match_full():
    q, k, v = rand_qkv(2, 4, 2, 64, 64, 64, seed=3)
    of, lf = oracle.attn(q, k, v, True)
    rows = [0, 5, 64 + 63, 3 * 64 + 17, 7 * 64 + 63]
    o, l = oracle.attn(q, k, v, True, rows=rows)
    np.testing.assert_array_equal(o, of.reshape(-1, 64)[rows])
    np.testing.assert_array_equal(l, lf.reshape(-1)[rows])


@pytest.mark.parametrize("Sq,Skv,causal", [(512, 512, False), (512, 512, True), (64, 200, True),
                                           (7, 7, True), (32768, 32768, True)])
def test_unmasked_pairs_closed_form(Sq, Skv, causal):
    n = oracle.unmasked_pairs(Sq, Skv, causal)
    if not causal:
        assert n == Sq * Skv
    elif Sq == Skv:
        assert n == Sq * (Sq + 1) // 2
    else:
        off = Skv - Sq
        assert n == sum(q + off + 1 for q in range(Sq))
    from long_context_sharded_gb300.workloads import unmasked_pairs
    assert unmasked_pairs(Sq, Skv, causal) == n
