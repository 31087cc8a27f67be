"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check that
the pins in test_oracle.py catch every one of them.

Each mutant is the oracle source with one edit, compiled to a temporary
library and loaded through MERCURY_ORACLE_LIB in a child pytest process.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle_attn.c")

MUTANTS = {
    "scale_1_over_d": ("1.0 / sqrt((double)d)", "1.0 / (double)d"),
    "gqa_map_modulo": ("int64_t g = h / G;", "int64_t g = h % Hkv;"),
    "causal_offset_dropped": ("int64_t lim = q + (Skv - Sq);", "int64_t lim = q;"),
    "shift_sign": ("s = (i + j) % R;", "s = (i + R - j) % R;"),
    "nested_levels_swapped": ("s = ((a + so) % Ro) * Ri + (b + t) % Ri;",
                              "s = ((a + t) % Ro) * Ri + (b + so) % Ri;"),
    "merge_weight_uses_max": ("double w = exp(lse_part[(int64_t)j * rows + r] - L);",
                              "double w = exp(lse_part[(int64_t)j * rows + r] - M);"),
    "value_uses_key_rows": ("o[t] += w * bf16_to_f64(vr[t]);", "o[t] += w * bf16_to_f64(kr[t]);"),
    "lse_drops_max": ("double L = M + log(Z);\n    for (int64_t c", "double L = log(Z);\n    for (int64_t c"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, "mutation site vanished: " + name
    if name == "value_uses_key_rows":
        src = src.replace("const uint16_t *vr = Vg + (k_lo + c) * (int64_t)d;",
                          "const uint16_t *vr = Vg + (k_lo + c) * (int64_t)d;\n"
                          "        const uint16_t *kr = Kg + (k_lo + c) * (int64_t)d; (void)vr;")
    src = src.replace(old, new)
    c_path = tmp_path / "mutant.c"
    c_path.write_text(src)
    so_path = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", str(c_path),
                    "-o", str(so_path), "-lm"], check=True)
    env = dict(os.environ, MERCURY_ORACLE_LIB=str(so_path))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, "mutant %s survived the pins:\n%s" % (name, r.stdout[-2000:])
