"""Work accounting for the throughput metric (FLOPs and algorithmic bytes).

The FLOP rule is the pages' own: each call counts the two matrix products Q K^T and
P V, 4 * B * Q * K * H * D, with multiply and add each one FLOP ("LingBot full-pipeline
analysis report", section "recorded cross-attention matrix work"), and K is the
*effective* (valid) length, never the allocated one (section "per-call effective
attention length": the allocated length overstates the work). The utilisation is the
effective FLOPs over (time x peak) (section "attention effective-FLOP utilisation
curve (A0)"). The backward counts 2.5 x the forward.

Here "effective" is exact: the number of (query, key) pairs that the mask leaves
visible, summed over batches and heads, so that causal rows count their own lengths.
"""

from __future__ import annotations

import numpy as np

__all__ = ["visible_pairs", "fwd_flops", "bwd_flops", "utilisation", "fwd_bytes",
           "bwd_bytes"]


def visible_pairs(B: int, Hq: int, Hkv: int, Sq: int, Skv: int, causal: bool,
                  kv_lens=None) -> int:
    """Number of visible (query, key) pairs summed over every (batch, query head)."""
    if kv_lens is None:
        lens = np.full((B, Hkv), Skv, dtype=np.int64)
    else:
        if hasattr(kv_lens, "detach"):
            kv_lens = kv_lens.detach().to("cpu").numpy()
        lens = np.asarray(kv_lens, dtype=np.int64).reshape(B, Hkv)
    g = Hq // Hkv
    total = 0
    for b in range(B):
        for kvh in range(Hkv):
            L = int(lens[b, kvh])
            if not causal:
                per = Sq * L
            else:
                # query i sees keys 0 .. min(L - 1, i + L - Sq)
                i = np.arange(Sq, dtype=np.int64)
                per = int(np.clip(i + L - Sq + 1, 0, L).sum())
            total += g * per
    return int(total)


def fwd_flops(B, Hq, Hkv, Sq, Skv, D, causal, kv_lens=None) -> float:
    return 4.0 * D * visible_pairs(B, Hq, Hkv, Sq, Skv, causal, kv_lens)


def bwd_flops(B, Hq, Hkv, Sq, Skv, D, causal, kv_lens=None) -> float:
    return 2.5 * fwd_flops(B, Hq, Hkv, Sq, Skv, D, causal, kv_lens)


def utilisation(flops: float, seconds: float, peak_flops_per_s: float) -> float:
    return flops / (seconds * peak_flops_per_s)


def fwd_bytes(B, Hq, Hkv, Sq, Skv, D, elem_bytes, kv_lens=None) -> float:
    """Algorithmic bytes of one forward: read Q, the valid K/V rows; write O and LSE."""
    if kv_lens is None:
        kv_rows = B * Hkv * Skv
    else:
        if hasattr(kv_lens, "detach"):
            kv_lens = kv_lens.detach().to("cpu").numpy()
        kv_rows = int(np.asarray(kv_lens, dtype=np.int64).sum())
    q_o = 2 * B * Sq * Hq * D * elem_bytes
    kv = 2 * kv_rows * D * elem_bytes
    lse = B * Hq * Sq * 4
    return float(q_o + kv + lse)


def bwd_bytes(B, Hq, Hkv, Sq, Skv, D, elem_bytes, kv_lens=None) -> float:
    """Algorithmic bytes of one backward: read Q, K, V, O, dO, LSE; write dQ, dK, dV."""
    if kv_lens is None:
        kv_rows = B * Hkv * Skv
    else:
        if hasattr(kv_lens, "detach"):
            kv_lens = kv_lens.detach().to("cpu").numpy()
        kv_rows = int(np.asarray(kv_lens, dtype=np.int64).sum())
    qsz = B * Sq * Hq * D * elem_bytes
    kvsz = kv_rows * D * elem_bytes
    return float(4 * qsz + 4 * kvsz + B * Hq * Sq * 4)
