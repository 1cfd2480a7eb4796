"""attn_fwd_decode_noalloc: the decode path for callers that cannot allocate
device memory at call time (their HBM is owned by another allocator, or they
cannot take the synchronisation an allocation may bring). It keeps the split
partials in a fixed library-owned device array instead of a workspace.

Collected last on purpose (file name), so a failure here never hides the
other tests. The GPU test calls the entry point through the C ABI twice in a
row, with different inputs, and holds each result to the float64 oracle with
the element-wise gate of the other parity tests, and to attn_fwd on the same
inputs. A second GPU test goes through the Python wrapper on a stream other
than the current one. Both also pass when run alone in a fresh process: the
first call looks up the scratch address itself.

The argument checks run in a child process that sees no GPU, with fake
device addresses: they must be rejected before anything touches CUDA, so a
regression that moved a check after a launch shows up there as
ATTN_ERR_CUDA instead of kernels reading unmapped memory.
"""

import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from exact_io_aware_attn_gb300 import _lib, build as build_mod
from exact_io_aware_attn_gb300.inputs import BF16, F16, make_qkv
from parity_helpers import LSE_TOL, O_TOL, compare, oracle_fwd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# Runs in a child with CUDA_VISIBLE_DEVICES="" and prints the statuses as JSON.
# Fake, aligned, far-apart addresses: validation never dereferences them.
_REJECTIONS = r"""
import json, sys
sys.path.insert(0, sys.argv[1])
from exact_io_aware_attn_gb300 import _lib
Q, K, V, O, LSE = ((1 << 40) * i for i in range(1, 6))
bf = _lib.ATTN_BF16
out = {
    # 32*12 rows x 1024 partitions x (128+4) floats = 207 MB > the 16 MiB scratch
    "oversized": _lib.fwd_decode_noalloc_raw(Q, K, V, O, LSE, 32, 12, 16384, 128, 0.088, bf,
                                             num_splits=1024),
    "null_q": _lib.fwd_decode_noalloc_raw(0, K, V, O, LSE, 2, 3, 100, 64, 0.125, bf),
    "d96": _lib.fwd_decode_noalloc_raw(Q, K, V, O, LSE, 2, 3, 100, 96, 0.125, bf),
    "neg_splits": _lib.fwd_decode_noalloc_raw(Q, K, V, O, LSE, 2, 3, 100, 64, 0.125, bf,
                                              num_splits=-1),
    "empty": _lib.fwd_decode_noalloc_raw(Q, K, V, O, LSE, 0, 3, 100, 64, 0.125, bf),
}
print(json.dumps(out))
"""


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return _lib.lib()


def test_argument_checks_run_before_any_cuda_call(lib):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", _REJECTIONS, ROOT], capture_output=True, text=True,
                       env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    st = json.loads(r.stdout.strip().splitlines()[-1])
    assert st["oversized"] == _lib.ATTN_ERR_WORKSPACE
    assert _lib.status_string(st["oversized"]) == "ATTN_ERR_WORKSPACE"
    assert st["null_q"] == _lib.ATTN_ERR_INVALID_ARG
    assert st["d96"] == _lib.ATTN_ERR_UNSUPPORTED
    assert st["neg_splits"] == _lib.ATTN_ERR_INVALID_ARG
    assert st["empty"] == _lib.ATTN_OK


def _check(o, lse, q, k, v, dtype, what):
    """o, lse: device results of the allocation-free call. Held to the
    oracle (element-wise gate) and to attn_fwd on the same inputs."""
    o_n = o.double().cpu().numpy()
    l_n = lse.double().cpu().numpy()
    compare(o_n, l_n, oracle_fwd(q.cpu(), k.cpu(), v.cpu(), causal=False), dtype, what)
    o_ref, lse_ref = _lib.attn_fwd(q, k, v)
    torch.cuda.synchronize()
    st, word = _lib.get_device_error()
    assert st == _lib.ATTN_OK, word
    assert np.abs(o_n - o_ref.double().cpu().numpy()).max() <= O_TOL, what
    assert np.abs(l_n - lse_ref.double().cpu().numpy()).max() <= LSE_TOL, what


def _noalloc_raw(B, h, T_kv, d, dtype, seed, num_splits):
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in make_qkv(B, h, 1, T_kv, d, dtype, seed=seed))
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, h, 1), float("nan"), dtype=torch.float32, device=dev)
    st = _lib.fwd_decode_noalloc_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                     lse.data_ptr(), B, h, T_kv, d, d ** -0.5, dtype, num_splits,
                                     torch.cuda.current_stream().cuda_stream)
    assert st == _lib.ATTN_OK, _lib.status_string(st)
    torch.cuda.synchronize()
    st, word = _lib.get_device_error()
    assert st == _lib.ATTN_OK, word
    _check(o, lse, q, k, v, dtype, f"noalloc B{B} h{h} Tkv{T_kv} d{d} splits={num_splits}")


@pytest.mark.gpu
def test_noalloc_matches_oracle_two_calls_in_a_row(lib, cuda_device):
    # the decode workload's shape with the library's split choice, then a
    # second call with other inputs, dtype, width and split count: the second
    # call reuses the shared scratch the first one left behind
    _noalloc_raw(32, 12, 16384, 64, BF16, seed=0, num_splits=0)
    _noalloc_raw(3, 5, 3001, 128, F16, seed=7, num_splits=13)


@pytest.mark.gpu
def test_noalloc_wrapper_on_a_side_stream(lib, cuda_device):
    # the Python wrapper, on a stream other than the current one: the call
    # is ordered on that stream alone
    q, k, v = (t.to(cuda_device) for t in make_qkv(4, 6, 1, 2500, 64, BF16, seed=5))
    o = torch.full_like(q, float("nan"))
    lse = torch.full((4, 6, 1), float("nan"), dtype=torch.float32, device=cuda_device)
    side = torch.cuda.Stream(device=cuda_device)
    side.wait_stream(torch.cuda.current_stream(cuda_device))
    _lib.attn_fwd_decode_noalloc(q, k, v, out=o, lse=lse, num_splits=7, stream=side)
    side.synchronize()
    _check(o, lse, q, k, v, BF16, "noalloc wrapper, side stream")
