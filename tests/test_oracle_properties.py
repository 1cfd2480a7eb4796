"""Property-based pins of the oracle (no GPU; needs hypothesis).

Random shapes, scales, block sizes and partition counts, with score ranges
wide enough that the running maximum moves many times: the block-wise
recurrence ("E8.1 IO-aware attention" Part 2, "IO-Aware Attention ...",
section "Softmax over blocks, exactly") and the partition merge (section
"Parallelism and the cost of the split") must both give the materialised
result, and a causal row must equal unmasked attention over its visible keys.
"""

import numpy as np
import pytest

import oracle

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")
given, settings = hyp.given, hyp.settings

ROW = st.tuples(
    st.integers(1, 40),            # keys
    st.integers(1, 9),             # d
    st.floats(0.05, 4.0),          # scale
    st.floats(0.1, 30.0),          # spread of the inputs (wide: the max moves often)
    st.integers(0, 2 ** 31 - 1),   # seed
)


def _row(n, d, spread, seed):
    rng = np.random.default_rng(seed)
    q = rng.normal(0.0, spread, d)
    k = rng.normal(0.0, 1.0, (n, d))
    v = rng.normal(0.0, 1.0, (n, d))
    return q, k, v


@settings(max_examples=150, deadline=None)
@given(ROW, st.integers(1, 45))
def test_blockwise_equals_materialised(row, block):
    n, d, scale, spread, seed = row
    q, k, v = _row(n, d, spread, seed)
    o_ref, lse_ref = oracle.standard_attention_row(q, k, v, scale=scale)
    o, m, l, _ = oracle.online_attention(q, k, v, block, scale=scale, return_state=True)
    np.testing.assert_allclose(o, o_ref, rtol=1e-9, atol=1e-12)
    lse = m + np.log(l)          # the recurrence's final state gives the row's lse
    assert abs(lse - lse_ref) <= 1e-9 * max(1.0, abs(lse_ref))


@settings(max_examples=150, deadline=None)
@given(ROW, st.integers(1, 50))
def test_partition_merge_equals_materialised(row, splits):
    n, d, scale, spread, seed = row
    q, k, v = _row(n, d, spread, seed)
    o_ref, lse_ref = oracle.standard_attention_row(q, k, v, scale=scale)
    o, lse = oracle.split_kv_attention(q, k, v, splits, scale=scale)
    np.testing.assert_allclose(o, o_ref, rtol=1e-9, atol=1e-12)
    assert abs(lse - lse_ref) <= 1e-9 * max(1.0, abs(lse_ref))


@settings(max_examples=80, deadline=None)
@given(st.integers(1, 12), st.integers(0, 12), st.integers(1, 6), st.integers(0, 2 ** 31 - 1))
def test_causal_row_is_attention_over_its_visible_keys(t_q, extra, d, seed):
    """Bottom-right alignment: row i of T_q rows against T_kv = T_q + extra
    keys sees exactly keys 0 .. i + extra."""
    t_kv = t_q + extra
    rng = np.random.default_rng(seed)
    q = rng.normal(size=(t_q, d))
    k = rng.normal(size=(t_kv, d))
    v = rng.normal(size=(t_kv, d))
    o, lse = oracle.standard_attention(q, k, v, scale=0.5, causal=True)
    for i in range(t_q):
        o_i, lse_i = oracle.standard_attention_row(q[i], k[:i + extra + 1], v[:i + extra + 1],
                                                   scale=0.5)
        np.testing.assert_allclose(o[i], o_i, rtol=1e-12, atol=1e-14)
        assert abs(lse[i] - lse_i) <= 1e-12 * max(1.0, abs(lse_i))
