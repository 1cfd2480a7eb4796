"""The oracle: a float64 CPU restatement of exact attention and its cost
model, written from the pages. TEST INFRASTRUCTURE ONLY: imported by the
tests, the smoke check and the benchmark's CPU-baseline leg, never by the
product path."""

from .oracle import (  # noqa: F401
    attention_backward,
    causal_visible,
    gqa_attention,
    gqa_attention_backward,
    merge_partials,
    online_attention,
    online_softmax_states,
    paged_decode_attention,
    split_kv_attention,
    split_partials,
    standard_attention,
    standard_attention_row,
)
from .cost import (  # noqa: F401
    attention_flops,
    attention_pairs,
    causal_pairs,
    kv_bytes,
    num_blocks,
    score_bytes,
    tile_bytes,
)
