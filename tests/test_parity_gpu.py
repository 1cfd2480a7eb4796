"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle
on the same seeded 16-bit inputs.

Small and medium shapes are compared element by element on every output;
the full-size workloads (in the launch configuration the benchmark times)
are compared on sampled rows the oracle computes one by one. Edge cases:
ragged tails, single tiles, T_q < T_kv under the causal mask, one key,
decode split counts that leave partitions empty, both dtypes, d = 64 and 128.
"""

import numpy as np
import pytest
import torch

from exact_io_aware_attn_gb300 import _lib
from exact_io_aware_attn_gb300.inputs import BF16, F16, WORKLOADS, make_qkv, make_workload
from parity_helpers import check_case, compare, gpu_fwd, oracle_fwd, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu(cuda_device):
    from exact_io_aware_attn_gb300 import build
    build.build()
    yield


# --------------------------------------------------------------- prefill
@pytest.mark.parametrize("shape", [
    # B, h, T_q, T_kv, d, dtype, causal
    (1, 2, 256, 256, 64, F16, False),       # the tiny exact-check workload, whole
    (2, 3, 1000, 1000, 64, BF16, True),     # GPT-2-shaped, ragged tail
    (1, 1, 128, 128, 64, BF16, True),       # exactly one tile
    (1, 1, 129, 129, 64, BF16, True),       # one row into a second tile
    (1, 1, 127, 127, 64, F16, False),
    (1, 1, 2, 2, 64, BF16, True),           # smallest prefill
    (1, 2, 300, 700, 64, BF16, False),      # T_q != T_kv, unmasked
    (1, 2, 300, 1000, 64, BF16, True),      # causal, bottom-right aligned
    (1, 1, 129, 4000, 128, F16, True),
    (1, 2, 640, 640, 128, BF16, True),      # d = 128
    (2, 2, 333, 333, 128, F16, False),
    (1, 1, 5, 1, 64, BF16, False),          # one key: O = V
    (3, 1, 384, 384, 64, F16, True),
    # at most 128 query rows at d = 64: two heads per unit (head-pair mode)
    (1, 3, 77, 77, 64, BF16, True),         # odd head count: the last unit has one head
    (2, 2, 128, 128, 64, F16, False),
    (1, 5, 2, 700, 64, BF16, False),        # two rows against a longer context
    (2, 3, 100, 300, 64, F16, True),        # bottom-right causal mask, six heads
])
def test_prefill_matches_oracle(shape):
    B, h, tq, tk, d, dt, causal = shape
    check_case(B, h, tq, tk, d, dt, causal)


@pytest.mark.parametrize("mult,dt", [(0.5, F16), (3.0, BF16), (3.0, F16)])
def test_prefill_input_scales(mult, dt):
    # x0.5: near-uniform rows (the very-long workload's recipe);
    # x3: very peaked rows whose running max moves often (exercises rescaling)
    check_case(1, 2, 1000, 1000, 64, dt, True, mult=mult, seed=3)
    check_case(1, 1, 700, 700, 128, dt, False, mult=mult, seed=4)


def test_prefill_other_scale():
    check_case(1, 2, 500, 500, 64, BF16, True, scale=0.3)
    check_case(1, 2, 500, 500, 128, F16, False, scale=0.02)


# --------------------------------------------------------------- decode
@pytest.mark.parametrize("splits", [None, 1, 7, 16, 32, 64])
def test_decode_split_counts(splits):
    check_case(2, 3, 1, 1000, 64, BF16, False, num_splits=splits)


@pytest.mark.parametrize("shape", [
    (1, 1, 1, 1, 64, BF16, False, None),     # one key
    (1, 2, 1, 5, 64, BF16, False, 16),       # more partitions than keys: empty ones
    (2, 2, 1, 777, 128, F16, False, None),
    (2, 2, 1, 777, 128, BF16, False, 13),
    (1, 3, 1, 4097, 64, F16, False, 64),
    (2, 2, 1, 300, 64, BF16, True, None),    # causal: one query sees the whole cache
])
def test_decode_matches_oracle(shape):
    B, h, tq, tk, d, dt, causal, splits = shape
    check_case(B, h, tq, tk, d, dt, causal, num_splits=splits)


def test_decode_result_independent_of_split_count():
    q, k, v = make_qkv(4, 3, 1, 3000, 64, BF16, seed=5)
    outs = [gpu_fwd(q, k, v, False, num_splits=s) for s in (1, 3, 16, 64, 1024)]
    o0, l0 = outs[0]
    for o, lse in outs[1:]:
        # fp32 sums in another order may round to a neighbouring bf16 value
        assert (np.abs(o - o0) <= 2.0 ** -7 * np.abs(o0) + 1e-3).all()
        assert np.abs(lse - l0).max() <= 1e-5


# --------------------------------------------------------------- full-size workloads
@pytest.mark.parametrize("w", WORKLOADS, ids=lambda w: w.name)
def test_full_size_workload_sampled(w):
    q, k, v = make_workload(w)
    o, lse = gpu_fwd(q, k, v, w.causal)
    if w.T_q == 1:
        ref = oracle_fwd(q, k, v, w.causal)                     # every (b, h) row
        compare(o, lse, ref, w.dtype, w.name)
        return
    rows = sample_rows(w.T_q, seed=w.T_q)
    heads = sorted({(0, 0), (w.B - 1, w.h - 1), (w.B // 2, w.h // 2)})
    for b, hh in heads:
        sl = (slice(b, b + 1), slice(hh, hh + 1))
        ref = oracle_fwd(q[sl], k[sl], v[sl], w.causal, rows=rows)
        compare(o[sl][:, :, rows], lse[sl][:, :, rows], ref, w.dtype, f"{w.name} head ({b},{hh})")


# --------------------------------------------------------------- contract
def test_empty_call_writes_nothing():
    dev = torch.device("cuda:0")
    q = torch.zeros(0, 2, 16, 64, dtype=torch.bfloat16, device=dev)
    o, lse = _lib.attn_fwd(q, q, q)
    torch.cuda.synchronize()
    assert o.numel() == 0 and lse.numel() == 0


@pytest.mark.parametrize("T_q,T_kv", [(1, 2000), (300, 300)])
def test_outputs_stay_in_bounds(T_q, T_kv):
    """Canary regions after O and lse must stay untouched."""
    dev = torch.device("cuda:0")
    B, h, d = 2, 3, 64
    q, k, v = (t.to(dev) for t in make_qkv(B, h, T_q, T_kv, d, BF16, seed=9))
    n_o, n_l = B * h * T_q * d, B * h * T_q
    obuf = torch.full((n_o + 4096,), 7.0, dtype=torch.bfloat16, device=dev)
    lbuf = torch.full((n_l + 1024,), 7.0, dtype=torch.float32, device=dev)
    o = obuf[:n_o].view(B, h, T_q, d)
    lse = lbuf[:n_l].view(B, h, T_q)
    _lib.attn_fwd(q, k, v, causal=True, out=o, lse=lse)
    torch.cuda.synchronize()
    assert bool((obuf[n_o:] == 7.0).all())
    assert bool((lbuf[n_l:] == 7.0).all())
    assert bool(torch.isfinite(o.float()).all()) and bool(torch.isfinite(lse).all())


def test_deterministic():
    q, k, v = make_qkv(2, 2, 600, 600, 64, BF16, seed=11)
    a = gpu_fwd(q, k, v, True)
    b = gpu_fwd(q, k, v, True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_runs_on_a_side_stream():
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in make_qkv(1, 2, 512, 512, 64, BF16, seed=12))
    ref_o, ref_l = _lib.attn_fwd(q, k, v, causal=True)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o, lse = _lib.attn_fwd(q, k, v, causal=True)
    s.synchronize()
    torch.cuda.synchronize()
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_l)


def test_kernel_name_recorded():
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in make_qkv(1, 1, 256, 256, 64, BF16))
    _lib.attn_fwd(q, k, v)
    assert _lib.last_kernel_name() == "prefill_tcgen05_d64_bf16"
    _lib.attn_fwd(q[:, :, :1].contiguous(), k, v)
    assert _lib.last_kernel_name().startswith("decode_split_d64_bf16")


def test_linear_memory_for_very_long_sequence():
    """The 16,384-token workload needs no workspace at all; a decode call's
    workspace is a few floats per partition, never the score matrix."""
    assert _lib.workspace_bytes(1, 12, 16384, 16384, 64, 0) == 0
    score_bytes = 12 * 16384 * 16384 * 2
    assert _lib.workspace_bytes(32, 12, 1, 16384, 64, 0) < score_bytes // 1000
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    q, k, v = (t.to("cuda") for t in make_qkv(1, 12, 16384, 16384, 64, F16, 0.5))
    o = torch.empty_like(q)
    lse = torch.empty(1, 12, 16384, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    _lib.attn_fwd(q, k, v, causal=True, out=o, lse=lse)
    torch.cuda.synchronize()
    free2, _ = torch.cuda.mem_get_info()
    # no allocation beyond the caller's tensors (allow 64 MiB of driver noise)
    assert free1 - free2 < 64 << 20, (free0, free1, free2)
