"""The bounds-checked build (-DMERCURY_CHECK), the stand-in for a memory
checker on this library's kernels: every TMA coordinate and every output
index is tested before use, and a bad one is reported (MERCURY_EBOUNDS) and
skipped instead of touching memory.

Without a GPU: the variant compiles and exports every declared symbol.  On
the GPU: the small parity shapes run through it in a child process (the
binding picks the library when it is imported) with no report, results within
the parity tolerances of the oracle, and O and LSE bit-identical to the
normal build's (the checks add branches, not arithmetic)."""
import ctypes
import os
import subprocess
import sys

import pytest

from tests.conftest import ROOT


def test_checked_build_compiles_and_exports():
    from long_context_sharded_gb300 import build
    path = build.build(check=True)
    assert path == build.CHECK_LIB_PATH and os.path.exists(path)
    lib = ctypes.CDLL(path)
    from tests.test_abi import declared_symbols
    for name in declared_symbols():
        assert hasattr(lib, name), name


@pytest.mark.gpu
def test_small_shapes_clean_under_the_checked_build():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tempfile

    import numpy as np

    from long_context_sharded_gb300 import build
    from long_context_sharded_gb300 import mercury as m
    from long_context_sharded_gb300.inputs import make_qkv
    from tests.checked_run import SHAPES
    build.build(check=True)
    # the normal build's results, for the bit-for-bit comparison in the child
    ref = {}
    for i, cfg in enumerate(SHAPES):
        B, Hq, Hkv, Sq, Skv, d, R, shift, causal = cfg
        q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, d, seed=sum(cfg[:7]))
        out, lse = m.mercury_attn_sharded(q.cuda(), k.cuda(), v.cuda(), R, shift, causal)
        m.mercury_sync_status()
        ref["o%d" % i], ref["l%d" % i] = out.cpu().numpy(), lse.cpu().numpy()
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, "normal_build.npz")
        np.savez(path, **ref)
        env = dict(os.environ, MERCURY_CHECKED_BUILD="1")
        r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "checked_run.py"), path], env=env,
                           capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "bit-identical to the normal build" in r.stdout
    assert "checked build: all" in r.stdout
