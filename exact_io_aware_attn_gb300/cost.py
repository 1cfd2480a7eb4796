"""Algorithmic work of one attention forward, for throughput reporting.

FLOPs: each of the two products costs 2*d FLOPs per visible (query, key)
pair per head, 4*d in all ("Attention and Its Computational Cost",
section "What is being computed"); a causal mask keeps, for row i of T_q
rows against T_kv keys, the keys j <= i + T_kv - T_q.

Bytes: what the method must move at minimum -- Q, K, V read once, O written
once (16-bit) and the fp32 logsumexp written once. The score and
probability matrices are not counted: they never leave the chip.

Backward: the gradient products dV = P^T dO, dP = dO V^T, dQ = dS K and
dK = dS^T Q, plus recomputing S = Q K^T, are five products of 2*d FLOPs per
visible pair: 10*d per pair per head (2.5x the forward). Recomputing S a
second time, as a kernel that forms dQ apart from dK and dV does, is not
counted. Minimum bytes: Q, K, V, O, dO and lse read once, dQ, dK, dV written
once.
"""

from __future__ import annotations


def visible_pairs(T_q: int, T_kv: int, causal: bool) -> int:
    if not causal:
        return T_q * T_kv
    # rows i = 0..T_q-1 each see T_kv - T_q + i + 1 keys
    first = T_kv - T_q + 1
    return T_q * first + T_q * (T_q - 1) // 2


def flops(B: int, h: int, T_q: int, T_kv: int, d: int, causal: bool) -> int:
    return 4 * d * B * h * visible_pairs(T_q, T_kv, causal)


def min_bytes(B: int, h: int, T_q: int, T_kv: int, d: int, elem: int = 2, h_kv: int = 0) -> int:
    """h_kv: key/value heads under grouped-query attention (0 = h)."""
    qo = 2 * B * h * T_q * d * elem
    kv = 2 * B * (h_kv or h) * T_kv * d * elem
    lse = B * h * T_q * 4
    return qo + kv + lse


def kv_cache_bytes(B: int, h: int, T_kv: int, d: int, elem: int = 2) -> int:
    """The bytes a decode step must stream: every cached key and value."""
    return 2 * B * h * T_kv * d * elem


def bwd_flops(B: int, h: int, T_q: int, T_kv: int, d: int, causal: bool) -> int:
    return 10 * d * B * h * visible_pairs(T_q, T_kv, causal)


def bwd_min_bytes(B: int, h: int, T_q: int, T_kv: int, d: int, elem: int = 2, h_kv: int = 0) -> int:
    q_side = 4 * B * h * T_q * d * elem            # q, o, dO read; dQ written
    kv_side = 4 * B * (h_kv or h) * T_kv * d * elem  # k, v read; dK, dV written
    return q_side + kv_side + B * h * T_q * 4       # lse read
