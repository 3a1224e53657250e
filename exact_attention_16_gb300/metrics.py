"""Work accounting for the attention forward (no attention arithmetic).

The throughput metric counts only unmasked (query, key) pairs:
FLOPs = 4 * B * Hq * D * N_unmasked (two multiply-adds per pair and head
dimension: one in Q K^T, one in P V). With the bottom-right causal mask,
query i sees min(Sk, max(0, i + Sk - Sq + 1)) keys.
"""

from __future__ import annotations


def visible_keys(i: int, Sq: int, Sk: int, causal: bool) -> int:
    if not causal:
        return Sk
    return min(Sk, max(0, i + Sk - Sq + 1))


def unmasked_pairs(Sq: int, Sk: int, causal: bool) -> int:
    """Number of visible (i, j) pairs of one (batch, head), in closed form."""
    if not causal:
        return Sq * Sk
    off = Sk - Sq
    # rows with 0 < i + off + 1 < Sk see i + off + 1 keys; later rows see Sk
    lo = max(0, -off)                    # first row that sees a key
    hi = min(Sq, Sk - off)               # first row that sees every key (exclusive bound of the ramp)
    total = 0
    if hi > lo:
        a, b = lo + off + 1, (hi - 1) + off + 1
        total += (a + b) * (hi - lo) // 2
    total += max(0, Sq - max(hi, lo)) * Sk
    return total


def flops(B: int, Sq: int, Sk: int, Hq: int, D: int, causal: bool) -> int:
    return 4 * B * Hq * D * unmasked_pairs(Sq, Sk, causal)


def algorithmic_bytes(B: int, Sq: int, Sk: int, Hq: int, Hkv: int, D: int, elem: int = 2, lse: bool = True) -> int:
    """Q, K, V read once; O (and fp32 LSE) written once."""
    return elem * D * (2 * B * Sq * Hq + 2 * B * Sk * Hkv) + (4 * B * Hq * Sq if lse else 0)
