"""Failure detection on the GPU without a GPU fault.

Every device-side wait in the kernels is bounded. The self-test entry point
runs that same bounded wait on a barrier nothing completes, with a short
limit: it must give up, record ATTN_ERR_TIMEOUT (kernel 4, site 1) in the
device status word and return, leaving the context usable. No trap, no
fault, no hang.
"""

import time

import numpy as np
import pytest
import torch

from exact_io_aware_attn_gb300 import _lib, build as build_mod
from exact_io_aware_attn_gb300.inputs import BF16
from parity_helpers import check_case

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu(cuda_device):
    build_mod.build()
    st, _ = _lib.get_device_error()   # start from a clear status word
    assert st == _lib.ATTN_OK
    yield


def test_bounded_wait_times_out_and_reports():
    t0 = time.perf_counter()
    assert _lib.selftest_wait_timeout(20000) == _lib.ATTN_OK      # 20 ms limit
    st, word = _lib.get_device_error()
    elapsed = time.perf_counter() - t0
    assert st == _lib.ATTN_ERR_TIMEOUT
    assert word & 0xff == _lib.ATTN_ERR_TIMEOUT
    assert (word >> 8) & 0xff == 4          # the self-test kernel
    assert (word >> 16) & 0xff == 1         # its only wait site
    assert 0.015 < elapsed < 5.0            # it waited about the limit, then returned
    # reading cleared the word
    assert _lib.get_device_error() == (_lib.ATTN_OK, 0)


def test_first_error_wins():
    assert _lib.selftest_wait_timeout(5000) == _lib.ATTN_OK
    assert _lib.selftest_wait_timeout(5000) == _lib.ATTN_OK
    st, word = _lib.get_device_error()
    assert st == _lib.ATTN_ERR_TIMEOUT and (word >> 8) & 0xff == 4
    assert _lib.get_device_error() == (_lib.ATTN_OK, 0)


def test_context_usable_after_timeout():
    assert _lib.selftest_wait_timeout(5000) == _lib.ATTN_OK
    assert _lib.get_device_error()[0] == _lib.ATTN_ERR_TIMEOUT
    # prefill and decode still give the oracle's answer
    check_case(1, 2, 300, 300, 64, BF16, True)
    check_case(2, 2, 1, 700, 64, BF16, False)


def test_limit_out_of_range_rejected():
    assert _lib.selftest_wait_timeout(0) == _lib.ATTN_ERR_INVALID_ARG
    assert _lib.selftest_wait_timeout(2000001) == _lib.ATTN_ERR_INVALID_ARG
    assert _lib.get_device_error() == (_lib.ATTN_OK, 0)
