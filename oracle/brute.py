"""Independent numpy brute force for tiny inputs (test infrastructure only).

Written separately from ``oracle_attn.c`` to pin it: dense score matrix with
numpy, the mask built as a boolean matrix, exp taken directly without the max
subtraction (so only valid while scores stay small, which tiny test inputs
ensure), probabilities normalised by an explicit sum.  Same definition as the
pages' attention patch (plain softmax attention, Silicon & Systems "The tuning
bill": checks against single-device FlashAttention).
"""
from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    u32 = bits.astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, causal: bool):
    """q [B,Hq,Sq,d], k/v [B,Hkv,Skv,d] float64.  Returns (O, LSE)."""
    B, Hq, Sq, d = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    kk = np.repeat(k, G, axis=1)          # q head h -> kv head h // G
    vv = np.repeat(v, G, axis=1)
    s = np.einsum("bhqd,bhkd->bhqk", q, kk) / np.sqrt(d)
    qi = np.arange(Sq)[:, None]
    ki = np.arange(Skv)[None, :]
    allowed = np.ones((Sq, Skv), dtype=bool) if not causal else (ki <= qi + (Skv - Sq))
    e = np.where(allowed, np.exp(s), 0.0)
    z = e.sum(axis=-1)
    with np.errstate(divide="ignore", invalid="ignore"):
        p = e / z[..., None]
        o = np.einsum("bhqk,bhkd->bhqd", np.where(z[..., None] > 0, p, 0.0), vv)
        lse = np.log(z)
    return o, lse
