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
    assert _lib.last_kernel_name().startswith("decode_split_gqa_d128_bf16")
    b = [0, w.B - 1]
    ref = oracle_fwd_gqa(q[b], k[b], v[b], False)
    compare(o[b], lse[b], ref, w.dtype, w.name)
