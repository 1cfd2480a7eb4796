"""GPU parity of the backward pass (attn_bwd, attn_bwd_gqa) against the
oracle's attention_backward / gqa_attention_backward, element by element,
on the same 16-bit inputs. o and lse come from the library's own forward
(the pipeline a training step runs), except where noted.

Shapes span several 128-row resident tiles and 64-row streamed tiles with
ragged tails on both sides, causal and not, T_q < T_kv (bottom-right mask),
T_q > T_kv, one query row, d = 64 and 128, bf16 and fp16, and groups of 2,
3 and 8 query heads per key/value head."""

import numpy as np
import pytest
import torch

from exact_io_aware_attn_gb300 import _lib
from exact_io_aware_attn_gb300.inputs import BF16, F16, GPT2_PREFILL, make_dout, make_qkv
from parity_helpers import compare_grads, gpu_bwd, oracle_bwd, oracle_fwd

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu(cuda_device):
    from exact_io_aware_attn_gb300 import build
    build.build()
    yield


def _name(shape):
    return "x".join(str(int(s)) for s in shape)


CASES = [
    # B, h, T_q, T_kv, d, dtype, causal
    (1, 2, 256, 256, 64, BF16, False),
    (1, 2, 256, 256, 64, BF16, True),
    (1, 2, 200, 333, 64, F16, False),      # ragged on both sides
    (1, 2, 200, 333, 64, BF16, True),      # T_q < T_kv: bottom-right causal mask
    (2, 1, 130, 130, 128, BF16, True),     # one row past a tile
    (1, 2, 1, 77, 64, BF16, False),        # one query row
    (1, 1, 1, 300, 128, F16, True),        # one causal query sees every key
    (1, 1, 333, 129, 64, BF16, False),     # T_q > T_kv
    (1, 1, 1024, 1024, 64, BF16, True),    # eight resident tiles
    (1, 1, 640, 640, 128, F16, True),
    (1, 3, 64, 1000, 64, BF16, True),      # few rows against a long cache
    (1, 1, 5, 7, 128, BF16, False),        # tiny
    (1, 2, 1, 300, 64, BF16, True),        # one causal query row at d = 64
    (1, 1, 5, 7, 64, F16, False),          # tiny at d = 64
    (1, 2, 700, 900, 64, F16, True),       # several 128-row tiles, ragged on both sides
]


@pytest.mark.parametrize("case", CASES, ids=_name)
def test_backward_parity(case):
    B, h, T_q, T_kv, d, dt, causal = case
    q, k, v = make_qkv(B, h, T_q, T_kv, d, dt, seed=31)
    do = make_dout(B, h, T_q, d, dt, seed=31)
    got = gpu_bwd(q, k, v, do, causal)
    compare_grads(got, oracle_bwd(q, k, v, do, causal), dt, f"bwd {case}")


GQA_CASES = [
    # B, h_q, h_kv, T_q, T_kv, d, dtype, causal
    (1, 4, 2, 200, 200, 64, BF16, True),
    (2, 6, 2, 130, 257, 128, F16, False),  # group 3
    (1, 8, 1, 256, 256, 64, BF16, True),   # group 8: one CTA sums eight heads
    (1, 8, 2, 300, 500, 64, BF16, False),  # group 4, ragged, no mask
]


@pytest.mark.parametrize("case", GQA_CASES, ids=_name)
def test_backward_gqa_parity(case):
    B, hq, hkv, T_q, T_kv, d, dt, causal = case
    q, k, v = make_qkv(B, hq, T_q, T_kv, d, dt, seed=32, h_kv=hkv)
    do = make_dout(B, hq, T_q, d, dt, seed=32)
    got = gpu_bwd(q, k, v, do, causal)
    compare_grads(got, oracle_bwd(q, k, v, do, causal), dt, f"bwd gqa {case}")


def test_backward_non_default_scale():
    q, k, v = make_qkv(1, 2, 190, 190, 64, BF16, seed=33)
    do = make_dout(1, 2, 190, 64, BF16, seed=33)
    got = gpu_bwd(q, k, v, do, True, scale=0.05)
    compare_grads(got, oracle_bwd(q, k, v, do, True, scale=0.05), BF16, "bwd scale 0.05")


def test_backward_from_oracle_forward():
    """The backward kernels alone: o (rounded to 16 bits) and lse (fp32) come
    from the oracle instead of the library's forward."""
    q, k, v = make_qkv(1, 2, 300, 300, 64, BF16, seed=34)
    do = make_dout(1, 2, 300, 64, BF16, seed=34)
    o_ref, lse_ref, _ = oracle_fwd(q, k, v, True)
    o16 = torch.from_numpy(o_ref).to(torch.bfloat16)
    lse32 = torch.from_numpy(lse_ref).to(torch.float32)
    got = gpu_bwd(q, k, v, do, True, o_lse=(o16, lse32))
    compare_grads(got, oracle_bwd(q, k, v, do, True), BF16, "bwd from oracle o/lse")


def test_backward_is_deterministic_and_workspace_independent():
    q, k, v = make_qkv(1, 2, 400, 400, 64, BF16, seed=35)
    do = make_dout(1, 2, 400, 64, BF16, seed=35)
    a = gpu_bwd(q, k, v, do, True)
    b = gpu_bwd(q, k, v, do, True)
    nbytes = _lib.bwd_workspace_bytes(1, 2, 400, 400, 64)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    c = gpu_bwd(q, k, v, do, True, workspace=ws)
    for x, y, z in zip(a, b, c):
        assert np.array_equal(x, y) and np.array_equal(x, z)


def test_backward_rejects_short_workspace():
    q, k, v = (t.cuda() for t in make_qkv(1, 1, 100, 100, 64, BF16))
    o, lse = _lib.attn_fwd(q, k, v, causal=True)
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(_lib.AttnError) as e:
        _lib.attn_bwd(q, k, v, o, lse, torch.ones_like(q), causal=True, workspace=ws)
    assert e.value.status == _lib.ATTN_ERR_WORKSPACE


def test_backward_gpt2_shape_sampled_heads():
    """The GPT-2 prefill shape (B 8, h 12, T 1024, d 64, causal, bf16) in
    one call, as the benchmark runs it; four (b, h) heads checked in full
    against the oracle run on those heads alone."""
    w = GPT2_PREFILL
    q, k, v = make_qkv(w.B, w.h, w.T_q, w.T_kv, w.d, w.dtype, seed=36)
    do = make_dout(w.B, w.h, w.T_q, w.d, w.dtype, seed=36)
    got = gpu_bwd(q, k, v, do, True)
    for (b, hh) in ((0, 0), (3, 7), (5, 11), (7, 5)):
        sl = (slice(b, b + 1), slice(hh, hh + 1))
        ref = oracle_bwd(q[sl], k[sl], v[sl], do[sl], True)
        compare_grads(tuple(g[sl] for g in got), ref, w.dtype, f"gpt2 bwd head {(b, hh)}")


def test_backward_single_key():
    """One key: P = 1, so dQ = dK = 0 (up to the fp32 difference dP - D,
    formed in two summation orders) and dV = dO exactly."""
    q, k, v = make_qkv(1, 1, 1, 1, 64, BF16, seed=37)
    do = make_dout(1, 1, 1, 64, BF16, seed=37)
    dq, dk, dv = gpu_bwd(q, k, v, do, True)
    assert np.abs(dq).max() <= 1e-5 and np.abs(dk).max() <= 1e-5
    assert np.array_equal(dv, do.double().numpy())


def test_backward_empty_is_a_no_op():
    x = torch.empty(0, 2, 16, 64, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(0, 2, 16, dtype=torch.float32, device="cuda")
    dq, dk, dv = _lib.attn_bwd(x, x, x, x, lse, x)
    assert dq.numel() == 0 and _lib.last_kernel_name() == "none"


def test_backward_kernel_name():
    q, k, v = (t.cuda() for t in make_qkv(1, 1, 128, 128, 128, F16))
    o, lse = _lib.attn_fwd(q, k, v)
    _lib.attn_bwd(q, k, v, o, lse, torch.ones_like(q))
    torch.cuda.synchronize()
    assert _lib.last_kernel_name() == "bwd_prep+bwd_dkdv+bwd_dq_tcgen05_d128_f16"


@pytest.mark.parametrize("case", [
    # B, h, T, d, dtype, heads checked
    (1, 16, 4096, 128, BF16, ((0, 0), (0, 13))),
    (1, 8, 4096, 64, F16, ((0, 3),)),
])
def test_backward_long_sampled_heads(case):
    """Long causal backward in one call; whole heads checked against the
    oracle run on those heads alone (the oracle materialises T x T per head)."""
    B, h, T, d, dt, heads = case
    q, k, v = make_qkv(B, h, T, T, d, dt, seed=38)
    do = make_dout(B, h, T, d, dt, seed=38)
    got = gpu_bwd(q, k, v, do, True)
    for (b, hh) in heads:
        sl = (slice(b, b + 1), slice(hh, hh + 1))
        ref = oracle_bwd(q[sl], k[sl], v[sl], do[sl], True)
        compare_grads(tuple(g[sl] for g in got), ref, dt, f"long bwd {case[:5]} head {(b, hh)}")


def test_backward_gqa_moderate_size():
    """Grouped-query backward, 8 query heads on 2 key/value heads, T 1024:
    each dK/dV CTA sums four query heads' contributions."""
    q, k, v = make_qkv(2, 8, 1024, 1024, 64, BF16, seed=39, h_kv=2)
    do = make_dout(2, 8, 1024, 64, BF16, seed=39)
    got = gpu_bwd(q, k, v, do, True)
    compare_grads(got, oracle_bwd(q, k, v, do, True), BF16, "gqa bwd T1024")
