"""The small parity shapes through the bounds-checked build of the library.

Run by tests/test_checked_build.py in a child process with
MERCURY_CHECKED_BUILD=1, so the binding loads the variant compiled with
-DMERCURY_CHECK: its kernels test every TMA coordinate and output index and
report an out-of-range one as MERCURY_EBOUNDS instead of touching memory.
Every call here must give no such report and match the fp64 oracle with the
usual tolerances.  Prints one summary line and exits 0 on success.
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import oracle  # noqa: E402
from long_context_sharded_gb300 import mercury as m  # noqa: E402
from long_context_sharded_gb300.inputs import make_qkv  # noqa: E402

O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3

SHAPES = [
    # B, Hq, Hkv, Sq, Skv, d, R, shift, causal
    (1, 4, 4, 512, 512, 64, 4, 1, False),
    (2, 4, 2, 384, 384, 128, 3, 1, True),
    (1, 8, 1, 128, 4096, 128, 4, 1, False),
    (1, 8, 2, 96, 96, 64, 3, 1, True),
    (1, 3, 1, 200, 200, 128, 2, 1, True),
    (1, 6, 3, 64, 192, 128, 8, 2, True),
    (1, 2, 2, 1000, 1000, 128, 1, 1, True),
    (1, 8, 8, 1024, 1024, 128, 8, 4, True),
]


def close(o, l, o_ref, l_ref, what):
    o = np.asarray(o, np.float64).reshape(o_ref.shape)
    l = np.asarray(l, np.float64).reshape(l_ref.shape)
    fin = np.isfinite(l_ref)
    err = np.abs(o - o_ref)
    ok = (np.isfinite(o).all() and (np.isfinite(l) == fin).all() and err.max() <= O_MAX
          and err.mean() <= O_MEAN and (not fin.any() or np.abs(l[fin] - l_ref[fin]).max() <= LSE_MAX))
    if not ok:
        raise SystemExit("%s: O max %.3g mean %.3g" % (what, err.max(), err.mean()))


def compare_with_normal_build(path):
    """Bit-identical to the normal build: the checks add branches, no arithmetic."""
    ref = np.load(path)
    n = 0
    for i, cfg in enumerate(SHAPES):
        B, Hq, Hkv, Sq, Skv, d, R, shift, causal = cfg
        q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, d, seed=sum(cfg[:7]))
        out, lse = m.mercury_attn_sharded(q.cuda(), k.cuda(), v.cuda(), R, shift, causal)
        m.mercury_sync_status()
        if not (np.array_equal(out.cpu().numpy(), ref["o%d" % i]) and
                np.array_equal(lse.cpu().numpy(), ref["l%d" % i])):
            raise SystemExit("checked and normal builds differ on %s" % (cfg,))
        n += 1
    return n


def main():
    assert m.CHECKED, "MERCURY_CHECKED_BUILD=1 must select the checked library"
    if len(sys.argv) > 1:
        print("checked build: bit-identical to the normal build on %d shapes" % compare_with_normal_build(sys.argv[1]))
    n = 0
    for cfg in SHAPES:
        B, Hq, Hkv, Sq, Skv, d, R, shift, causal = cfg
        q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, d, seed=sum(cfg[:7]))
        qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
        o_ref, l_ref = oracle.attn(q, k, v, causal)
        out, lse = m.mercury_attn_sharded(qd, kd, vd, R, shift, causal)
        m.mercury_sync_status()
        close(out.cpu(), lse.cpu(), o_ref, l_ref, "sharded %s" % (cfg,))
        op, lp = m.mercury_attn_partial(qd, kd, vd, R, shift, causal)
        out, lse = m.mercury_lse_merge(op, lp)
        m.mercury_sync_status()
        close(out.cpu(), lse.cpu(), o_ref, l_ref, "partial+merge %s" % (cfg,))
        o16, l16 = m.mercury_attn_sharded_bf16(qd, kd, vd, R, shift, causal)
        m.mercury_sync_status()
        close(o16.float().cpu(), l16.cpu(), o_ref, l_ref, "bf16 %s" % (cfg,))
        if R >= 2:
            out, lse = m.mercury_attn_run_schedule(qd, kd, vd, causal, (R, R, 2, shift))
            m.mercury_sync_status()
            close(out.cpu(), lse.cpu(), o_ref, l_ref, "two runs %s" % (cfg,))
        n += 1
    q, k, v = make_qkv(2, 16, 4, 3, 4096, 128, seed=3)
    out, lse = m.mercury_attn_decode(q.cuda(), k.cuda(), v.cuda(), 0, False)
    m.mercury_sync_status()
    o_ref, l_ref = oracle.attn(q, k, v, False)
    close(out.cpu(), lse.cpu(), o_ref, l_ref, "decode")
    g = torch.Generator().manual_seed(7)
    a = torch.randn(384, 200, generator=g).bfloat16()
    b = torch.randn(200, 320, generator=g).bfloat16()
    c = m.mercury_gemm_shifted(a.cuda(), b.cuda(), 2, 1)
    m.mercury_sync_status()
    ref = a.double() @ b.double()
    err = (c.cpu().double() - ref).abs().max().item()
    if err > 1e-2:
        raise SystemExit("gemm: max err %.3g" % err)
    print("checked build: all %d shapes, decode and GEMM clean" % n)


if __name__ == "__main__":
    main()
