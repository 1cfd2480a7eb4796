"""attn_fwd_decode_noalloc: the decode path for callers that cannot allocate
device memory at call time (their HBM is owned by another allocator, or they
cannot take the synchronisation an allocation may bring). It keeps the split
partials in a fixed library-owned device array instead of a workspace.

Collected last on purpose (file name), so a failure here never hides the
other tests. The GPU test calls the entry point through the C ABI twice in a
row, with different inputs, and compares each result with attn_fwd on the
same inputs, within the parity tolerances used by the other GPU tests. It
also passes when run alone in a fresh process: the first call sets up the
scratch address itself.
"""

import numpy as np
import pytest
import torch

from exact_io_aware_attn_gb300 import _lib, build as build_mod
from exact_io_aware_attn_gb300.inputs import BF16, F16, make_qkv
from parity_helpers import LSE_TOL, O_TOL

# fake, aligned, far-apart addresses: validation never dereferences them
Q, K, V, O, LSE = ((1 << 40) * i for i in range(1, 6))


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return _lib.lib()


def test_oversized_request_rejected_before_launch(lib):
    # 32*12 rows x 1024 partitions x (128+4) floats = 207 MB > the 16 MiB scratch
    st = _lib.fwd_decode_noalloc_raw(Q, K, V, O, LSE, 32, 12, 16384, 128, 0.088, _lib.ATTN_BF16,
                                     num_splits=1024)
    assert st == _lib.ATTN_ERR_WORKSPACE
    assert _lib.status_string(st) == "ATTN_ERR_WORKSPACE"


def test_invalid_arguments_rejected(lib):
    assert _lib.fwd_decode_noalloc_raw(0, K, V, O, LSE, 2, 3, 100, 64, 0.125,
                                       _lib.ATTN_BF16) == _lib.ATTN_ERR_INVALID_ARG
    assert _lib.fwd_decode_noalloc_raw(Q, K, V, O, LSE, 2, 3, 100, 96, 0.125,
                                       _lib.ATTN_BF16) == _lib.ATTN_ERR_UNSUPPORTED
    assert _lib.fwd_decode_noalloc_raw(Q, K, V, O, LSE, 2, 3, 100, 64, 0.125, _lib.ATTN_BF16,
                                       num_splits=-1) == _lib.ATTN_ERR_INVALID_ARG
    assert _lib.fwd_decode_noalloc_raw(Q, K, V, O, LSE, 0, 3, 100, 64, 0.125,
                                       _lib.ATTN_BF16) == _lib.ATTN_OK      # empty


def _noalloc_vs_fwd(B, h, T_kv, d, dtype, seed, num_splits):
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in make_qkv(B, h, 1, T_kv, d, dtype, seed=seed))
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, h, 1), float("nan"), dtype=torch.float32, device=dev)
    st = _lib.fwd_decode_noalloc_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                     lse.data_ptr(), B, h, T_kv, d, d ** -0.5, dtype, num_splits,
                                     torch.cuda.current_stream().cuda_stream)
    assert st == _lib.ATTN_OK, _lib.status_string(st)
    o_ref, lse_ref = _lib.attn_fwd(q, k, v)
    torch.cuda.synchronize()
    st, word = _lib.get_device_error()
    assert st == _lib.ATTN_OK, word
    o_n, o_r = o.double().cpu().numpy(), o_ref.double().cpu().numpy()
    l_n, l_r = lse.double().cpu().numpy(), lse_ref.double().cpu().numpy()
    assert np.isfinite(o_n).all() and np.isfinite(l_n).all()
    assert np.abs(o_n - o_r).max() <= O_TOL
    assert np.abs(l_n - l_r).max() <= LSE_TOL


@pytest.mark.gpu
def test_noalloc_matches_attn_fwd_two_calls_in_a_row(lib, cuda_device):
    # the decode workload's shape with the library's split choice, then a
    # second call with other inputs, dtype, width and split count: the second
    # call reuses the shared scratch the first one left behind
    _noalloc_vs_fwd(32, 12, 16384, 64, BF16, seed=0, num_splits=0)
    _noalloc_vs_fwd(3, 5, 3001, 128, F16, seed=7, num_splits=13)
