"""The C ABI without a GPU: the library loads and exports every declared
symbol, the shift planner matches the hand-written tables and the oracle's
independent table, argument validation rejects bad calls before any CUDA
call, and the work decomposition covers every output exactly once."""
import ctypes
import os
import re

import numpy as np
import pytest

from tests.conftest import ROOT, load_golden_table


@pytest.fixture(scope="module")
def m():
    from long_context_sharded_gb300 import build
    build.build()
    from long_context_sharded_gb300 import mercury
    return mercury


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "mercury_attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mercury_\w+)\s*\(", text)))


def test_library_exports_every_declared_symbol(m):
    names = declared_symbols()
    assert len(names) >= 8
    for name in names:
        assert hasattr(m.lib, name), name
    assert sorted(m.EXPORTED) == names


def test_no_oracle_in_product_package():
    pkg = os.path.join(ROOT, "long_context_sharded_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".h", ".cuh", ".cpp")):
                src = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert "import oracle" not in src and "from oracle" not in src, f
                assert "oracle_attn" not in src, f


@pytest.mark.parametrize("R,shift,name", [(4, 1, "shift_R4_flat.txt"),
                                          (4, 0, "shift_R4_unshifted.txt"),
                                          (8, 4, "shift_R8_nested_2x4.txt")])
def test_plan_shift_golden(m, R, shift, name):
    assert m.mercury_plan_shift(R, shift).tolist() == load_golden_table(name)


@pytest.mark.parametrize("R", [1, 2, 3, 4, 5, 8, 12, 16, 64, 128])
def test_plan_shift_matches_oracle_and_is_latin(m, R):
    import oracle
    for shift in [0, 1] + [k for k in range(2, R + 1) if R % k == 0]:
        t = m.mercury_plan_shift(R, shift)
        assert (t == oracle.shift_order(R, shift)).all()
        if shift:
            for i in range(R):
                assert sorted(t[i]) == list(range(R))
                assert sorted(t[:, i]) == list(range(R))


@pytest.mark.parametrize("R,shift", [(0, 1), (129, 1), (8, 3), (8, -1), (6, 4)])
def test_plan_shift_rejects(m, R, shift):
    buf = np.zeros(max(R * R, 1), np.int32)
    rc = m.lib.mercury_plan_shift(R, shift, buf.ctypes.data_as(ctypes.c_void_p))
    assert rc == m.MERCURY_EINVAL
    assert m.lib.mercury_last_error()


GOOD = dict(B=1, Hq=4, Hkv=2, Sq=256, Skv=256, d=128, R=4, shift=1, causal=0)
P = 0x100000  # fake, 16-byte aligned "device" address: validation never dereferences


def call(m, fn="mercury_attn_sharded", q=P, k=P, v=P, out=P, lse=P, **kw):
    a = dict(GOOD, **kw)
    return getattr(m.lib, fn)(q, k, v, a["B"], a["Hq"], a["Hkv"], a["Sq"], a["Skv"], a["d"],
                              a["R"], a["shift"], a["causal"], out, lse, None)


@pytest.mark.parametrize("fn", ["mercury_attn_sharded", "mercury_attn_partial"])
@pytest.mark.parametrize("kw,code", [
    (dict(q=0), -1), (dict(k=0), -1), (dict(v=0), -1), (dict(out=0), -1), (dict(lse=0), -1),
    (dict(d=96), -1), (dict(d=256), -1), (dict(Hq=6, Hkv=4), -1), (dict(Sq=250), -1),
    (dict(Skv=130), -1), (dict(R=0), -1), (dict(R=256, Sq=256 * 2, Skv=256 * 2), -1),
    (dict(shift=3), -1), (dict(shift=-2), -1), (dict(causal=1, Sq=512, Skv=256), -1),
    (dict(B=0), -1), (dict(Hkv=0), -1), (dict(Sq=0), -1),
    (dict(q=P + 2), -2), (dict(k=P + 8), -2), (dict(v=P + 4), -2), (dict(out=P + 4), -2),
    (dict(lse=P + 2), -2),
])
def test_attention_argument_validation(m, fn, kw, code):
    assert call(m, fn, **kw) == code
    assert m.lib.mercury_last_error()


@pytest.mark.parametrize("args,code", [
    ((0, P, 4, 10, 128, P, P), -1), ((P, 0, 4, 10, 128, P, P), -1), ((P, P, 0, 10, 128, P, P), -1),
    ((P, P, 4097, 10, 128, P, P), -1), ((P, P, 4, -1, 128, P, P), -1), ((P, P, 4, 10, 6, P, P), -1),
    ((P, P, 4, 10, 0, P, P), -1), ((P, P, 4, 10, 516, P, P), -1), ((P + 4, P, 4, 10, 128, P, P), -2),
    ((P, P, 4, 10, 128, P + 8, P), -2), ((P, P + 2, 4, 10, 128, P, P), -2),
    ((P, P, 4, 1 << 60, 128, P, P), -1),
])
def test_merge_argument_validation(m, args, code):
    assert m.lib.mercury_lse_merge(*args, None) == code


def call_noalloc(m, q=P, k=P, v=P, out=P, lse=P, n_runs=2, **kw):
    a = dict(GOOD, **kw)
    return m.lib.mercury_attn_split_noalloc(q, k, v, a["B"], a["Hq"], a["Hkv"], a["Sq"], a["Skv"], a["d"],
                                            a["R"], a["shift"], a["causal"], n_runs, out, lse, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), -1), (dict(k=0), -1), (dict(v=0), -1), (dict(out=0), -1), (dict(lse=0), -1),
    (dict(d=96), -1), (dict(n_runs=0), -1), (dict(n_runs=5), -1), (dict(R=0), -1), (dict(R=129), -1),
    (dict(shift=3), -1), (dict(causal=1, Sq=512, Skv=256), -1), (dict(Sq=250), -1), (dict(Hq=6, Hkv=4), -1),
    (dict(q=P + 2), -2), (dict(k=P + 8), -2), (dict(v=P + 4), -2), (dict(out=P + 4), -2), (dict(lse=P + 2), -2),
])
def test_noalloc_argument_validation(m, kw, code):
    """The allocation-free entry point rejects bad arguments before any CUDA
    call (so these run without a GPU)."""
    assert call_noalloc(m, **kw) == code
    assert m.lib.mercury_last_error()


@pytest.mark.parametrize("n_runs", [64, 8])
def test_noalloc_rejects_partials_beyond_its_array(m, n_runs):
    # n_runs x 8*2048 rows x (128+1) x 4 bytes: 541 MB and 68 MB, both over 64 MiB
    rc = call_noalloc(m, B=1, Hq=8, Hkv=1, Sq=2048, Skv=8192, d=128, R=64, n_runs=n_runs)
    assert rc == m.MERCURY_EINVAL
    msg = m.lib.mercury_last_error()
    assert b"scratch" in msg and b"67108864" in msg


def test_merge_zero_rows_is_noop(m):
    assert m.lib.mercury_lse_merge(P, P, 4, 0, 128, P, P, None) == 0


WORKLOAD_GEOMS = {
    # name: (Mq, Gp, head_mode)
    "mha_b1_h4_d64_s512_r4": (128, 1, 0),
    "gqa_b1_hq32_hkv8_d128_s32k_causal_r8": (128, 1, 1),
    "mha_b16_h32_d128_s4k_r8": (128, 1, 0),
    "gqa_b1_hq64_hkv8_d128_s128k_causal_r8_nested2x4": (128, 1, 1),
    "mqa_b1_hq8_hkv1_d128_sq2k_skv2m_r64_merge": (32, 4, 1),
}


@pytest.mark.parametrize("name", sorted(WORKLOAD_GEOMS))
def test_workload_geometry(m, name):
    from long_context_sharded_gb300.workloads import WORKLOADS
    w = WORKLOADS[name]
    info = m.mercury_work_decomposition(w["B"], w["Hq"], w["Hkv"], w["Sq"], w["Skv"], w["d"],
                                        w["R"], w["causal"], 1 if w["mode"] == "partial" else 0)
    assert (info["Mq"], info["Gp"], info["head_mode"]) == WORKLOAD_GEOMS[name]
    assert info["n_items"] < 2 ** 31


COVERAGE = [
    # B, Hq, Hkv, Sq, Skv, d, R, shift, causal
    (1, 4, 4, 512, 512, 64, 4, 1, 0),
    (2, 4, 2, 256, 256, 128, 2, 1, 1),
    (1, 8, 1, 128, 4096, 128, 4, 1, 0),      # Bq = 32: heads packed 4 per tile
    (1, 8, 2, 96, 96, 64, 3, 1, 1),          # Bq = 32, G = 4
    (1, 3, 1, 200, 200, 128, 2, 0, 1),       # odd group, ragged block
    (2, 2, 2, 384, 384, 64, 3, 1, 0),        # MHA row pairs with odd tile count
    (1, 6, 3, 64, 192, 128, 8, 2, 1),        # Bq = 8, Sq < Skv causal, nested
]


def _random_coverage_shapes(n, seed):
    """Seeded shapes within the call's contract (head packing, ragged blocks and
    shards, GQA groups, causal with Sq <= Skv, every shift form)."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        R = int(rng.choice([1, 2, 3, 4, 5, 8, 16]))
        Hkv = int(rng.choice([1, 2, 3]))
        G = int(rng.choice([1, 2, 4, 8]))
        Sq = R * int(rng.integers(1, 80))
        Skv = Sq if rng.random() < 0.5 else R * int(rng.integers(1, 120))
        causal = int(rng.random() < 0.5 and Sq <= Skv)
        shifts = [0, 1] + [k for k in range(2, R) if R % k == 0]
        out.append((int(rng.choice([1, 2])), Hkv * G, Hkv, Sq, Skv, int(rng.choice([64, 128])), R,
                    int(rng.choice(shifts)), causal))
    return out


COVERAGE += _random_coverage_shapes(10, 7)


@pytest.mark.parametrize("cfg", COVERAGE)
@pytest.mark.parametrize("mode", [0, 1, 2, 3, 5])
def test_work_items_cover_each_output_once(m, cfg, mode):
    B, Hq, Hkv, Sq, Skv, d, R, shift, causal = cfg
    if mode > R:
        pytest.skip("more runs than steps")
    info = m.mercury_work_decomposition(B, Hq, Hkv, Sq, Skv, d, R, causal, mode)
    slots = info["slots"]
    if mode == 0:
        assert slots == 1
    elif mode == 1:
        assert slots == R
    else:
        spg = -(-R // mode)
        assert slots == -(-R // spg) and slots <= mode
    seen = {}
    for item in range(info["n_items"]):
        rows, step = m.mercury_work_item_rows(B, Hq, Hkv, Sq, Skv, d, R, shift, causal, mode, item)
        assert len(rows) <= 256
        if mode:
            assert 0 <= step < slots
        else:
            assert step == -1
        for r in rows:
            key = (r, step)
            assert key not in seen, "row %d slot %d written twice" % key
            seen[key] = item
    expect = B * Hq * Sq * (slots if mode else 1)
    assert len(seen) == expect
    partial = mode == 1
    if partial:
        # the item writing (row, step j) reads shard order[rank][j]
        order = m.mercury_plan_shift(R, shift)
        Bq = Sq // R
        for (r, j) in list(seen)[:2000]:
            assert 0 <= order[(r % Sq) // Bq][j] < R
