"""The five synthetic workloads, named by what they are.

They stand in for the pages' Llama-3-like MHA / GQA attention workloads
(batch 1 and 16, contexts from 4K to 2M tokens; Silicon & Systems, "What
Mercury finds that templates miss").  No dataset or trained weights are used:
Q, K, V are seeded N(0, 1) * scale, rounded to bf16 (see ``inputs.py``).

``shift``: 0 unshifted, 1 flat (i + j) mod R, k >= 2 nested with inner size k.
``mode``: "fused" runs the online accumulator across all steps in one kernel;
"partial" emits one (O, LSE) pair per step and merges them afterwards.
"""
from __future__ import annotations

WORKLOADS = {
    "mha_b1_h4_d64_s512_r4": dict(
        B=1, Hq=4, Hkv=4, Sq=512, Skv=512, d=64, causal=False, R=4, shift=1,
        scale=1.0, seed=1, mode="fused"),
    "gqa_b1_hq32_hkv8_d128_s32k_causal_r8": dict(
        B=1, Hq=32, Hkv=8, Sq=32768, Skv=32768, d=128, causal=True, R=8, shift=1,
        scale=0.5, seed=2, mode="fused"),
    "mha_b16_h32_d128_s4k_r8": dict(
        B=16, Hq=32, Hkv=32, Sq=4096, Skv=4096, d=128, causal=False, R=8, shift=1,
        scale=1.0, seed=3, mode="fused"),
    "gqa_b1_hq64_hkv8_d128_s128k_causal_r8_nested2x4": dict(
        B=1, Hq=64, Hkv=8, Sq=131072, Skv=131072, d=128, causal=True, R=8, shift=4,
        scale=0.5, seed=4, mode="fused"),
    "mqa_b1_hq8_hkv1_d128_sq2k_skv2m_r64_merge": dict(
        B=1, Hq=8, Hkv=1, Sq=2048, Skv=2097152, d=128, causal=False, R=64, shift=1,
        scale=1.0, seed=5, mode="partial"),
}

# The workload the throughput benchmark times: the largest that fits one GPU
# (Llama-3-70B-like GQA, 128K context, nested 2 x 4 shift).
BENCH_WORKLOAD = "gqa_b1_hq64_hkv8_d128_s128k_causal_r8_nested2x4"
# The small workload every check can run in full on the CPU oracle.
SMALL_WORKLOAD = "mha_b1_h4_d64_s512_r4"


def unmasked_pairs(Sq: int, Skv: int, causal: bool) -> int:
    """Unmasked (query, key) pairs for one (batch, head): key k is allowed for
    query q iff k <= q + (Skv - Sq) under the causal mask."""
    if not causal:
        return Sq * Skv
    off = Skv - Sq
    total = 0
    # rows with q + off >= Skv - 1 see every key; the rest see q + off + 1 keys
    full_from = max(0, Skv - 1 - off)
    n_full = max(0, Sq - full_from)
    total += n_full * Skv
    # q in [max(0, -off), full_from): q + off + 1 keys each
    lo = max(0, -off)
    hi = min(full_from, Sq)
    if hi > lo:
        a = lo + off + 1
        b = hi - 1 + off + 1
        total += (a + b) * (hi - lo) // 2
    return total


def attention_flops(w: dict) -> int:
    """Algorithmic FLOPs: 4*d per unmasked (q, k) pair (2*d for the score, 2*d
    for the value sum), over all batches and query heads."""
    return 4 * w["d"] * w["B"] * w["Hq"] * unmasked_pairs(w["Sq"], w["Skv"], w["causal"])


# The all-gather GEMM pattern (the pages' second operator family, batch 16):
# a Llama-3-70B-like MLP projection, 16 x 1024 tokens x 8192 hidden -> 28672,
# R = 8 virtual ranks each owning a row block of A, B cut into 8 column shards.
GEMM_WORKLOADS = {
    "gemm_m16k_k8k_n28k_r8": dict(M=16384, K=8192, N=28672, R=8, shift=1, seed=6),
}
