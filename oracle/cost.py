"""Closed-form cost model of attention: TEST INFRASTRUCTURE ONLY.

Part of the oracle (see oracle/oracle.py): only the tests, the smoke check
and the benchmark's CPU-baseline leg may import it. The product package keeps
its own, independently written counter for the benchmark; the tests compare
the two.

Pages followed:

* "E8.1 IO-aware attention" (coursefy.online), "Part 2. Do it in code":
  score_bytes(n, bytes_per_value=2) is the size of an n x n score matrix,
  tile_bytes(t, bytes_per_value=2) of a t x t tile, num_blocks(n, block) is
  ceil(n / block).
* "Attention and Its Computational Cost" (programmer.ie, Inference ch. 8),
  section "What is being computed": each of the two products costs
  2 T_q T_kv d per head, 4 B h T_q T_kv d in all; causal self-attention over
  T tokens needs T(T+1)/2 of the T^2 pairs. Section "The other shape": a KV
  cache holds a key and a value vector per layer, head and position; the
  formula display was lost in extraction and is restated here as
  2 * layers * heads * T * d * bytes (it reproduces the printed 36 MiB per
  sequence at 1,024 tokens for GPT-2 small and the per-layer decode table).
"""

from __future__ import annotations

__all__ = [
    "score_bytes",
    "tile_bytes",
    "num_blocks",
    "causal_pairs",
    "attention_pairs",
    "attention_flops",
    "kv_bytes",
]


def score_bytes(n: int, bytes_per_value: int = 2) -> int:
    """Bytes of one n x n score matrix ("E8.1", Part 2)."""
    return n * n * bytes_per_value


def tile_bytes(t: int, bytes_per_value: int = 2) -> int:
    """Bytes of one t x t score tile ("E8.1", Part 2)."""
    return t * t * bytes_per_value


def num_blocks(n: int, block: int) -> int:
    """Number of key blocks of size `block` covering n keys: ceil(n/block)."""
    if block < 1:
        raise ValueError("block must be at least 1")
    return -(-n // block)


def causal_pairs(t: int) -> int:
    """Query-key pairs a causal mask keeps over t tokens: t(t+1)/2."""
    return t * (t + 1) // 2


def attention_pairs(q_len: int, kv_len: int, causal: bool) -> int:
    """Visible (query, key) pairs per head.

    Dense: q_len * kv_len. Causal with bottom-right alignment (row i sees
    keys j <= i + kv_len - q_len): q_len*(kv_len - q_len) + q_len(q_len+1)/2,
    which is causal_pairs(T) when q_len == kv_len == T.
    """
    if not causal:
        return q_len * kv_len
    if q_len > kv_len:
        raise ValueError("causal attention needs q_len <= kv_len")
    return q_len * (kv_len - q_len) + causal_pairs(q_len)


def attention_flops(batch: int, heads: int, q_len: int, kv_len: int,
                    head_dim: int, causal: bool = False) -> int:
    """FLOPs of the two products: 4 * head_dim per visible pair, per head.

    "Attention and Its Computational Cost", section "What is being
    computed" (2 T_q T_kv d per product; causal counts T(T+1)/2 pairs).
    """
    return 4 * batch * heads * head_dim * attention_pairs(q_len, kv_len, causal)


def kv_bytes(layers: int, heads: int, seq_len: int, head_dim: int,
             bytes_per_value: int = 2, batch: int = 1) -> int:
    """Bytes of a KV cache: one key and one value vector per layer, head,
    position and sequence ("Attention and Its Computational Cost", section
    "The other shape: one query, many keys")."""
    return 2 * layers * heads * seq_len * head_dim * bytes_per_value * batch
