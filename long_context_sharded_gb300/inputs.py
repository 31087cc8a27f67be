"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds none of the attention arithmetic: it only draws random
numbers and rounds them to bf16, so that the CUDA path and the CPU oracle are
fed the very same host bytes.

Recipe: ``torch.Generator('cpu').manual_seed(seed)``; draw ``randn`` in fp32 in
the order Q, K, V (each tensor in one call); multiply by ``scale``; round to
bf16 with round-to-nearest-even (torch's default cast).
"""
from __future__ import annotations

import torch


def make_qkv(B: int, Hq: int, Hkv: int, Sq: int, Skv: int, d: int,
             seed: int, scale: float = 1.0):
    """Return (q, k, v) as contiguous bf16 CPU tensors.

    q: [B, Hq, Sq, d]; k, v: [B, Hkv, Skv, d]."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    out = []
    for shape in ((B, Hq, Sq, d), (B, Hkv, Skv, d), (B, Hkv, Skv, d)):
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if scale != 1.0:
            x.mul_(scale)
        out.append(x.to(torch.bfloat16).contiguous())
        del x
    return tuple(out)


def sample_rows(B: int, Hq: int, Sq: int, R: int, seed: int,
                n_heads: int = 8, n_random: int = 256):
    """Seeded row sample for parity checks at full size.

    For a seeded subset of ``n_heads`` (b, h) pairs (all of them when there are
    fewer): rows 0, 1, every query-block start and end +-1, the last row, plus
    ``n_random`` seeded random rows.  Returns sorted unique flat row indices
    (b*Hq + h)*Sq + q."""
    g = torch.Generator(device="cpu").manual_seed(int(seed) + 7919)
    n_bh = B * Hq
    if n_bh <= n_heads:
        heads = torch.arange(n_bh)
    else:
        heads = torch.randperm(n_bh, generator=g)[:n_heads]
    Bq = Sq // R
    fixed = {0, 1, Sq - 1, Sq - 2}
    for i in range(R):
        for q in (i * Bq - 1, i * Bq, i * Bq + 1, (i + 1) * Bq - 2, (i + 1) * Bq - 1):
            if 0 <= q < Sq:
                fixed.add(q)
    rows = set()
    for bh in heads.tolist():
        for q in fixed:
            rows.add(bh * Sq + q)
        rnd = torch.randint(0, Sq, (n_random,), generator=g)
        for q in rnd.tolist():
            rows.add(bh * Sq + q)
    return sorted(rows)
