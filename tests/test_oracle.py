"""The oracle against its pins (CPU only).

Every check comes from tests/oracle_pins.py and compares the oracle with
something other than itself: the pages' worked example, a brute force, a
library routine, closed forms, invariants and the exactness of blocking.
"""

import math

import numpy as np
import pytest

import oracle
from oracle_pins import ALL_CHECKS, real_oracle


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    fails = check(real_oracle())
    assert not fails, fails


def test_block_below_one_is_value_error():
    q = np.ones(4)
    k = np.ones((3, 4))
    with pytest.raises(ValueError):
        oracle.online_attention(q, k, k, 0)
    with pytest.raises(ValueError):
        oracle.online_softmax_states([1.0, 2.0], 0)


def test_worked_example_values():
    # m and l after each block of 4 for the page's scores, to more digits
    states = oracle.online_softmax_states([1, 3, 2, 5, 4, 0, 6, 2], 4)
    assert states[0][0] == 5.0
    assert math.isclose(states[0][1], 1.2034380, rel_tol=1e-7)
    assert states[1][0] == 6.0
    assert math.isclose(states[1][1], 1.5988498, rel_tol=1e-7)
    # lse of the row = m + ln l
    assert math.isclose(6.0 + math.log(states[1][1]), 6.4692845, rel_tol=1e-7)


def test_causal_needs_tq_le_tkv():
    q = np.ones((4, 2))
    k = np.ones((3, 2))
    with pytest.raises(ValueError):
        oracle.standard_attention(q, k, k, causal=True)


def test_empty_partition_has_zero_weight():
    rng = np.random.default_rng(0)
    q = rng.standard_normal(4)
    k = rng.standard_normal((3, 4))
    v = rng.standard_normal((3, 4))
    ms, ls, os_ = oracle.split_partials(q, k, v, 5)   # chunk 1: splits 3, 4 empty
    assert np.isneginf(ms[3]) and ls[3] == 0.0 and not os_[3].any()
    o, lse = oracle.merge_partials(ms, ls, os_)
    o_ref, lse_ref = oracle.standard_attention_row(q, k, v)
    assert np.allclose(o, o_ref, rtol=1e-12) and math.isclose(lse, lse_ref, rel_tol=1e-12)


def test_fully_uniform_row_lse_is_log_count():
    # near-uniform rows (small inputs, as in the x0.5 workload) have lse ~ ln(#keys)
    t = 64
    q = np.zeros((t, 8))
    k = np.ones((t, 8))
    v = np.ones((t, 8))
    _, lse = oracle.standard_attention(q, k, v, causal=True)
    assert np.allclose(lse, np.log(np.arange(1, t + 1)), rtol=1e-13)
