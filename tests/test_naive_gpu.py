"""The materialising baseline (attn_fwd_naive): S and P written to device
memory, then O = P V -- the standard attention the IO-aware kernels are
measured against ("Attention and Its Computational Cost", section "The cost
of writing down the scores"; "E8.1 IO-aware attention" Part 2,
standard_attention).

GPU tests hold it to the float64 oracle on the same seeded 16-bit inputs:
plain and causal (bottom-right) shapes, ragged tiles, odd key counts (the
scalar paths), both widths and both dtypes. O is held to the stated
max |dO| <= 2e-2. This path stores each score in the 16-bit type before the
softmax (as a 16-bit framework's materialised score tensor is), so a score s
carries a relative error up to the unit roundoff u (2^-8 bf16, 2^-11 fp16)
and lse = ln sum exp(s) moves by at most u * max|s|: the lse gate is the
stated 1e-3 plus that amount. The element-wise rounding gate of the IO-aware
kernels does not apply.
CPU tests check the workspace size and the argument checks, which run before
any CUDA call (here in a child process that sees no GPU).
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
from parity_helpers import LSE_TOL, O_TOL, UNIT_ROUNDOFF, oracle_fwd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return _lib.lib()


def test_workspace_is_two_16bit_matrices(lib):
    assert _lib.naive_workspace_bytes(2, 3, 100, 200) == 2 * 2 * 3 * 100 * 200 * 2
    assert _lib.naive_workspace_bytes(1, 12, 16384, 16384) == 4 * 12 * 16384 * 16384
    assert _lib.naive_workspace_bytes(-1, 3, 100, 200) == 0


_CHECKS = r"""
import json, sys
sys.path.insert(0, sys.argv[1])
from exact_io_aware_attn_gb300 import _lib
Q, K, V, O, LSE, WS = ((1 << 40) * i for i in range(1, 7))
bf = _lib.ATTN_BF16
need = _lib.naive_workspace_bytes(2, 3, 100, 200)
out = {
    "heads": _lib.naive_raw(Q, K, V, O, LSE, 2, 40000, 100, 200, 64, 0.125, 1, bf, WS, 1 << 40),
    "short": _lib.naive_raw(Q, K, V, O, LSE, 2, 3, 100, 200, 64, 0.125, 1, bf, WS, need - 16),
    "misaligned": _lib.naive_raw(Q, K, V, O, LSE, 2, 3, 100, 200, 64, 0.125, 1, bf, WS + 8, need),
    "overlap": _lib.naive_raw(Q, K, V, O, LSE, 2, 3, 100, 200, 64, 0.125, 1, bf, Q, need),
    "d96": _lib.naive_raw(Q, K, V, O, LSE, 2, 3, 100, 200, 96, 0.125, 1, bf, WS, need),
    "causal_tall": _lib.naive_raw(Q, K, V, O, LSE, 2, 3, 300, 200, 64, 0.125, 1, bf, WS, need),
    "empty": _lib.naive_raw(Q, K, V, O, LSE, 0, 3, 100, 200, 64, 0.125, 1, bf, None, 0),
}
print(json.dumps(out))
"""


def test_argument_checks_before_any_cuda_call(lib):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", _CHECKS, ROOT], capture_output=True, text=True,
                       env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    st = json.loads(r.stdout.strip().splitlines()[-1])
    assert st["heads"] == _lib.ATTN_ERR_UNSUPPORTED
    assert st["short"] == _lib.ATTN_ERR_WORKSPACE
    assert st["misaligned"] == _lib.ATTN_ERR_WORKSPACE
    assert st["overlap"] == _lib.ATTN_ERR_WORKSPACE
    assert st["d96"] == _lib.ATTN_ERR_UNSUPPORTED
    assert st["causal_tall"] == _lib.ATTN_ERR_INVALID_ARG
    assert st["empty"] == _lib.ATTN_OK


def max_abs_score(q, k, causal):
    """max |scale * q_i . k_j| over the visible pairs, float64."""
    d = q.shape[-1]
    sc = (q.double() @ k.double().transpose(-1, -2)) * d ** -0.5
    if causal:
        T_q, T_kv = q.shape[-2], k.shape[-2]
        vis = torch.arange(T_kv)[None, :] <= torch.arange(T_q)[:, None] + (T_kv - T_q)
        sc = sc.masked_fill(~vis, 0.0)
    return float(sc.abs().max())


CASES = [
    # B, h, T_q, T_kv, d, dtype, causal, mult
    (1, 2, 256, 256, 64, F16, False, 1.0),      # the tiny workload
    (2, 3, 300, 700, 64, BF16, True, 1.0),      # bottom-right causal, ragged tiles
    (1, 1, 129, 129, 64, F16, True, 1.0),       # one row past a tile
    (1, 2, 1000, 1000, 128, BF16, True, 1.0),   # d = 128
    (2, 2, 1, 777, 64, BF16, False, 1.0),       # one query row, odd key count
    (1, 3, 200, 301, 128, F16, False, 1.0),     # odd key count, d = 128
    (1, 12, 2048, 2048, 64, F16, True, 0.5),    # the very long workload's heads, shorter
]


@pytest.mark.gpu
@pytest.mark.parametrize("B,h,T_q,T_kv,d,dtype,causal,mult", CASES)
def test_naive_matches_oracle(lib, cuda_device, B, h, T_q, T_kv, d, dtype, causal, mult):
    q, k, v = make_qkv(B, h, T_q, T_kv, d, dtype, mult, seed=11)
    qd, kd, vd = q.to(cuda_device), k.to(cuda_device), v.to(cuda_device)
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((B, h, T_q), float("nan"), dtype=torch.float32, device=cuda_device)
    ws = torch.empty(_lib.naive_workspace_bytes(B, h, T_q, T_kv), dtype=torch.uint8,
                     device=cuda_device)
    _lib.attn_fwd_naive(qd, kd, vd, causal=causal, out=o, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    st, word = _lib.get_device_error()
    assert st == _lib.ATTN_OK, word
    assert _lib.last_kernel_name().startswith("naive_scores+naive_softmax+naive_pv")
    o_ref, lse_ref, _ = oracle_fwd(q, k, v, causal)
    o_n, l_n = o.double().cpu().numpy(), lse.double().cpu().numpy()
    assert np.isfinite(o_n).all() and np.isfinite(l_n).all()
    assert np.abs(o_n - o_ref).max() <= O_TOL
    assert np.abs(l_n - lse_ref).max() <= LSE_TOL + UNIT_ROUNDOFF[dtype] * max_abs_score(q, k, causal)
    # the materialised matrices are really there: P rows sum to one
    n = B * h * T_q * T_kv
    p = ws[2 * n:4 * n].view(q.dtype).view(B, h, T_q, T_kv).double()
    assert torch.allclose(p.sum(-1), torch.ones_like(p.sum(-1)), atol=0.02)


@pytest.mark.gpu
def test_naive_without_caller_workspace(lib, cuda_device):
    q, k, v = (t.to(cuda_device) for t in make_qkv(1, 2, 500, 500, 64, BF16, seed=12))
    o, lse = _lib.attn_fwd_naive(q, k, v, causal=True)
    torch.cuda.synchronize()
    o_ref, lse_ref, _ = oracle_fwd(q.cpu(), k.cpu(), v.cpu(), True)
    assert np.abs(o.double().cpu().numpy() - o_ref).max() <= O_TOL
    assert (np.abs(lse.double().cpu().numpy() - lse_ref).max()
            <= LSE_TOL + UNIT_ROUNDOFF[BF16] * max_abs_score(q.cpu(), k.cpu(), True))
