"""GPU parity of grouped-query attention (query head i uses key/value head
i // (h_q / h_kv)) against the oracle's gqa_attention, through the C ABI
entry attn_fwd_gqa: decode (one CTA serves up to 8 query heads of a group,
reading each cached row once) and prefill (the unit's K/V loads use the
group's key/value head)."""

import pytest

from exact_io_aware_attn_gb300 import _lib
from exact_io_aware_attn_gb300.inputs import BF16, DECODE_GQA, F16, make_qkv, make_workload
from parity_helpers import compare, gpu_fwd_gqa, oracle_fwd_gqa, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu(cuda_device):
    from exact_io_aware_attn_gb300 import build
    build.build()
    yield


@pytest.mark.parametrize("shape", [
    # B, h_q, h_kv, T_q, T_kv, d, dtype, causal, splits
    (2, 8, 2, 1, 1000, 64, BF16, False, 0),     # group 4
    (1, 16, 2, 1, 3001, 64, BF16, False, 0),    # group 8
    (2, 6, 3, 1, 700, 64, F16, False, 7),       # group 2
    (1, 12, 1, 1, 2000, 64, BF16, False, 0),    # group 12: 3 CTAs of 4 heads per kv head
    (1, 9, 3, 1, 500, 128, BF16, False, 0),     # group 3: one head per CTA
    (2, 8, 1, 1, 1500, 128, F16, False, 16),    # group 8, d = 128
    (2, 8, 8, 1, 900, 64, BF16, False, 0),      # group 1: plain attention
    (1, 4, 2, 1, 5, 64, BF16, False, 16),       # more partitions than keys
])
def test_gqa_decode(shape):
    B, hq, hkv, tq, tk, d, dt, causal, splits = shape
    q, k, v = make_qkv(B, hq, tq, tk, d, dt, seed=21, h_kv=hkv)
    o, lse = gpu_fwd_gqa(q, k, v, causal, splits)
    compare(o, lse, oracle_fwd_gqa(q, k, v, causal), dt, f"gqa decode {shape}")


@pytest.mark.parametrize("shape", [
    (1, 8, 2, 500, 500, 64, BF16, True),
    (2, 4, 1, 300, 700, 64, F16, True),
    (1, 4, 2, 333, 333, 128, BF16, False),
    (1, 6, 3, 640, 640, 128, F16, True),
])
def test_gqa_prefill(shape):
    B, hq, hkv, tq, tk, d, dt, causal = shape
    q, k, v = make_qkv(B, hq, tq, tk, d, dt, seed=22, h_kv=hkv)
    o, lse = gpu_fwd_gqa(q, k, v, causal)
    compare(o, lse, oracle_fwd_gqa(q, k, v, causal), dt, f"gqa prefill {shape}")


def test_gqa_decode_full_size():
    w = DECODE_GQA
    q, k, v = make_workload(w)
    o, lse = gpu_fwd_gqa(q, k, v, False)
    # a group of 4 query heads per key/value head: the tensor-core path
    assert _lib.last_kernel_name().startswith("prefill_splitkv_tcgen05_d128_bf16")
    b = [0, w.B - 1]
    ref = oracle_fwd_gqa(q[b], k[b], v[b], False)
    compare(o[b], lse[b], ref, w.dtype, w.name)


@pytest.mark.parametrize("shape", [
    # B, h_q, h_kv, T_kv, d, dtype, splits -- groups >= 4 run as a prefill of
    # G query rows per key/value head on the tensor cores, then the merge
    (2, 8, 2, 3000, 64, BF16, 0),       # group 4
    (1, 16, 2, 5000, 128, BF16, 0),     # group 8
    (2, 12, 1, 700, 64, F16, 5),        # group 12
    (1, 16, 1, 129, 128, F16, 1),       # group 16, one partition: the plain kernel writes o
    (3, 8, 2, 1, 64, BF16, 0),          # a single key
    (1, 32, 8, 16384, 128, BF16, 64),   # the most partitions
    (3, 8, 1, 1000, 64, BF16, 0),       # three key/value heads: two in a unit, one alone
    (1, 4, 1, 500, 64, F16, 1),         # one key/value head: no pair, one partition
    (5, 4, 1, 2500, 64, BF16, 9),       # pairs across sequences, nine partitions
])
def test_gqa_decode_tensor_core_path(shape):
    B, hq, hkv, tk, d, dt, splits = shape
    q, k, v = make_qkv(B, hq, 1, tk, d, dt, seed=23, h_kv=hkv)
    o, lse = gpu_fwd_gqa(q, k, v, False, splits)
    assert _lib.last_kernel_name().startswith("prefill_")
    compare(o, lse, oracle_fwd_gqa(q, k, v, False), dt, f"gqa decode tc {shape}")


def test_gqa_decode_tensor_core_caller_workspace():
    import numpy as np
    import torch
    q, k, v = make_qkv(2, 8, 1, 2000, 128, BF16, seed=24, h_kv=2)
    dev = torch.device("cuda:0")
    nbytes = _lib.gqa_workspace_bytes(2, 8, 2, 1, 2000, 128, 6)
    assert nbytes == 2 * 8 * 6 * 132 * 4
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o1 = torch.empty_like(qd)
    l1 = torch.empty(2, 8, 1, dtype=torch.float32, device=dev)
    st = _lib.fwd_gqa_raw(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o1.data_ptr(), l1.data_ptr(),
                          2, 8, 2, 1, 2000, 128, 128 ** -0.5, 0, _lib.ATTN_BF16, 6, ws.data_ptr(),
                          nbytes, None)
    assert st == _lib.ATTN_OK
    o2, l2 = gpu_fwd_gqa(q, k, v, False, 6)
    assert np.array_equal(o1.double().cpu().numpy(), o2) and np.array_equal(l1.double().cpu().numpy(), l2)
    st = _lib.fwd_gqa_raw(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o1.data_ptr(), l1.data_ptr(),
                          2, 8, 2, 1, 2000, 128, 128 ** -0.5, 0, _lib.ATTN_BF16, 6, ws.data_ptr(),
                          nbytes - 16, None)
    assert st == _lib.ATTN_ERR_WORKSPACE
