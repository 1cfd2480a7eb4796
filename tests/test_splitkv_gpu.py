"""GPU parity of the split-KV prefill (attn_fwd_splitkv, and attn_fwd's own
choice to split small problems) against the oracle: the key range of every
pair of query tiles is cut into partitions whose fp32 partials the merge
kernel combines per query row.

Cases: short queries against a long causal context (the chunked-prefill
shape), non-causal, ragged query and key tails, more partitions than key
tiles (empty partitions), grouped-query heads, d = 64 and 128, bf16 and
fp16, automatic and fixed partition counts, caller and library workspace,
more units than SMs, and a caller workspace holding stale bytes."""

import numpy as np
import pytest
import torch

from exact_io_aware_attn_gb300 import _lib
from exact_io_aware_attn_gb300.inputs import BF16, F16, make_qkv
from parity_helpers import compare, oracle_fwd, oracle_fwd_gqa

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu(cuda_device):
    from exact_io_aware_attn_gb300 import build
    build.build()
    yield


def gpu_splitkv(q, k, v, causal, num_splits, workspace=None):
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.full_like(qd, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device=dev)
    _lib.attn_fwd_splitkv(qd, kd, vd, causal=causal, out=o, lse=lse, num_splits=num_splits,
                          workspace=workspace)
    torch.cuda.synchronize()
    st, word = _lib.get_device_error()
    assert st == _lib.ATTN_OK, f"device status {st} word {word:#x}"
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


CASES = [
    # B, h_q, h_kv, T_q, T_kv, d, dtype, causal, splits
    (1, 4, 4, 256, 4096, 64, BF16, True, 0),       # chunked prefill: 256 rows, long context
    (1, 4, 4, 256, 4096, 64, BF16, True, 7),
    (1, 2, 2, 300, 2000, 128, F16, False, 5),      # ragged query and key tails
    (1, 2, 2, 130, 300, 64, BF16, True, 8),        # more partitions than key tiles
    (2, 8, 2, 128, 3000, 64, BF16, True, 0),       # grouped-query, group 4
    (1, 3, 1, 2, 1000, 128, BF16, True, 4),        # two query rows
    (1, 1, 1, 512, 512, 64, F16, True, 3),         # causal square: early pairs see few tiles
    (1, 2, 2, 200, 8192, 128, BF16, False, 64),    # the most partitions
    (1, 8, 8, 1024, 2048, 128, BF16, True, 8),     # more units than SMs: CTAs loop, then merge
    (1, 6, 6, 100, 5000, 64, F16, False, 16),      # head pairs (d 64, one query tile)
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(str(int(x)) for x in c))
def test_splitkv_parity(case):
    B, hq, hkv, tq, tk, d, dt, causal, splits = case
    q, k, v = make_qkv(B, hq, tq, tk, d, dt, seed=51, h_kv=hkv)
    o, lse = gpu_splitkv(q, k, v, causal, splits)
    ref = oracle_fwd(q, k, v, causal) if hq == hkv else oracle_fwd_gqa(q, k, v, causal)
    compare(o, lse, ref, dt, f"splitkv {case}")


def test_attn_fwd_splits_small_problems_by_itself():
    """attn_fwd on a small-batch, long-context prefill picks partitions
    (kernel name) and matches the oracle; the unsplit prefill through
    attn_fwd_ex matches too."""
    q, k, v = make_qkv(1, 2, 256, 4096, 64, BF16, seed=52)
    dev = torch.device("cuda:0")
    o, lse = _lib.attn_fwd(q.to(dev), k.to(dev), v.to(dev), causal=True)
    torch.cuda.synchronize()
    assert _lib.last_kernel_name().startswith("prefill_splitkv_tcgen05_d64_bf16")
    ref = oracle_fwd(q, k, v, True)
    compare(o.double().cpu().numpy(), lse.double().cpu().numpy(), ref, BF16, "attn_fwd split")
    ws = torch.empty(64, dtype=torch.uint8, device=dev)
    o2, lse2 = _lib.attn_fwd(q.to(dev), k.to(dev), v.to(dev), causal=True, num_splits=0,
                             workspace=ws)
    torch.cuda.synchronize()
    assert _lib.last_kernel_name() == "prefill_tcgen05_d64_bf16"
    compare(o2.double().cpu().numpy(), lse2.double().cpu().numpy(), ref, BF16, "attn_fwd_ex")


def test_splitkv_caller_workspace_gives_the_same_bits():
    q, k, v = make_qkv(1, 4, 200, 3000, 128, F16, seed=53)
    a = gpu_splitkv(q, k, v, True, 6)
    nbytes = _lib.splitkv_workspace_bytes(1, 4, 200, 3000, 128, 6)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    b = gpu_splitkv(q, k, v, True, 6, workspace=ws)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_splitkv_one_partition_is_the_plain_kernel():
    q, k, v = make_qkv(1, 2, 256, 1024, 64, BF16, seed=54)
    o, lse = gpu_splitkv(q, k, v, True, 1)
    assert _lib.last_kernel_name() == "prefill_tcgen05_d64_bf16"
    compare(o, lse, oracle_fwd(q, k, v, True), BF16, "splitkv S=1")


def test_splitkv_ignores_stale_workspace_bytes():
    """A caller workspace filled with 0xff bytes, then the same workspace
    reused, give the oracle's result with the same bits: nothing the call
    reads from the workspace comes from an earlier call."""
    q, k, v = make_qkv(1, 4, 256, 6000, 64, BF16, seed=55)
    nbytes = _lib.splitkv_workspace_bytes(1, 4, 256, 6000, 64, 9)
    ws = torch.full((nbytes,), 255, dtype=torch.uint8, device="cuda")
    a = gpu_splitkv(q, k, v, True, 9, workspace=ws)
    assert _lib.last_kernel_name() == "prefill_splitkv_tcgen05_d64_bf16+decode_combine"
    compare(a[0], a[1], oracle_fwd(q, k, v, True), BF16, "split-KV, stale workspace")
    b = gpu_splitkv(q, k, v, True, 9, workspace=ws)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
