"""Work and traffic counts for the attention forward (measurement only).

FLOPs are mask-adjusted: every visible (query, key) pair costs 2*d flops for
its score (one d-long dot product) and 2*d for its share of P V, so
4*d per pair.  The algorithmic byte count is the traffic a fused forward cannot
avoid: Q, K and V read once, O and the per-row logsumexp written once; the
S x S score and probability matrices never reach memory ("FlashAttention:
IO-aware attention kernels", table "What goes in, what comes out").
"""
from __future__ import annotations


def visible_pairs_closed_form(Sq: int, Sk: int, mask: str, window: int = 0) -> int:
    """Number of visible (query, key) pairs per head, by counting formula.

    none: Sq*Sk.  causal (key j <= row i, j < Sk): sum_i min(i+1, Sk).
    window W (i-W < j <= i, j < Sk): sum_i (min(i, Sk-1) - max(0, i-W+1) + 1)^+.
    """
    if mask == "none":
        return Sq * Sk
    if mask == "causal":
        n = min(Sq, Sk)
        return n * (n + 1) // 2 + max(0, Sq - Sk) * Sk
    # window: split rows by which bound is active
    total = 0
    W = int(window)
    # rows i < Sk: count = min(i, W-1) + 1
    r1 = min(Sq, Sk)
    a = min(r1, W)            # rows 0..a-1 have i+1 keys
    total += a * (a + 1) // 2
    total += max(0, r1 - a) * W
    # rows i >= Sk: keys in [max(0,i-W+1), Sk-1]
    for i in range(Sk, Sq):
        lo = max(0, i - W + 1)
        total += max(0, Sk - lo)
    return total


def attention_flops(w) -> float:
    """Mask-adjusted forward FLOPs: 4*d per visible pair (QK^T and PV MACs x2)."""
    return 4.0 * w.d * w.B * w.H * visible_pairs_closed_form(w.Sq, w.Sk, w.mask, w.window)


def attention_bwd_flops(w) -> float:
    """Mask-adjusted backward FLOPs: 10*d per visible pair, the five tile
    products of the backward (S again, dV, dP, dQ, dK), i.e. 2.5x the forward.
    (The kernels form S and dP twice, 14*d per pair; the rate counts the
    algorithm's 10*d.)"""
    return 2.5 * attention_flops(w)


def bwd_algorithmic_bytes(w) -> int:
    """Bytes the backward must move at minimum: read Q, K, V, O, dO, lse and
    write dQ, dK, dV (the per-row statistics workspace excluded)."""
    e = 2
    hkv = getattr(w, "kv_heads", w.H)
    return (e * w.B * w.H * w.Sq * w.d * 3          # Q, O, dO
            + e * w.B * hkv * w.Sk * w.d * 2        # K, V
            + 4 * w.B * w.H * w.Sq                  # lse
            + e * w.B * w.H * w.Sq * w.d            # dQ
            + e * w.B * hkv * w.Sk * w.d * 2)       # dK, dV


def algorithmic_bytes(w) -> int:
    """Bytes the fused forward must move at minimum: read Q,K,V once, write O, lse."""
    e = 2
    hkv = getattr(w, "kv_heads", w.H)                        # K/V heads (grouped-query)
    return (e * w.B * (w.H * w.Sq * w.d + 2 * hkv * w.Sk * w.d)   # Q, K, V
            + e * w.B * w.H * w.Sq * w.d                      # O
            + 4 * w.B * w.H * w.Sq)                           # lse fp32
