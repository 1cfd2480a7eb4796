"""GPU parity of the host-buffer entry attn_fwd_host: q, k, v, o and lse in
host memory, the copies made by the library in stream order. Checked against
the oracle element by element and bit for bit against the device-pointer
path (the same kernels run on the device copies).

Cases: a causal grouped-query prefill and a decode (T_q = 1) against a
ragged cache, bf16 and fp16, d = 64 and 128; pinned and pageable host
buffers; the library's own device region and a caller's; a caller region
one byte short."""

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


CASES = [
    # B, h_q, h_kv, T_q, T_kv, d, dtype, causal, pinned, caller_buffer
    (1, 4, 2, 300, 300, 64, BF16, True, True, False),     # prefill, ragged tail, GQA
    (2, 4, 4, 1, 1000, 128, F16, False, True, True),      # decode, caller region
    (1, 2, 2, 256, 640, 64, F16, True, False, False),     # pageable host buffers
]


def _device_ref(q, k, v, causal):
    dev = torch.device("cuda:0")
    o, lse = _lib.attn_fwd_gqa(q.to(dev), k.to(dev), v.to(dev), causal=causal)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(str(int(x)) for x in c))
def test_host_entry_parity(case):
    B, hq, hkv, tq, tk, d, dt, causal, pinned, caller = case
    q, k, v = make_qkv(B, hq, tq, tk, d, dt, seed=71, h_kv=hkv)
    if pinned:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    buf = None
    if caller:
        buf = torch.empty(_lib.host_buffer_bytes(B, hq, hkv, tq, tk, d), dtype=torch.uint8,
                          device="cuda")
    o, lse = _lib.attn_fwd_host(q, k, v, causal=causal, device_buffer=buf)
    st, word = _lib.get_device_error()
    assert st == _lib.ATTN_OK, f"device status {st} word {word:#x}"
    ref = oracle_fwd(q, k, v, causal) if hq == hkv else oracle_fwd_gqa(q, k, v, causal)
    compare(o.double().numpy(), lse.double().numpy(), ref, dt, f"host entry {case}")
    o_dev, lse_dev = _device_ref(q, k, v, causal)
    assert torch.equal(o, o_dev) and torch.equal(lse, lse_dev)


def test_host_entry_short_buffer():
    q, k, v = make_qkv(1, 2, 128, 128, 64, BF16, seed=72)
    need = _lib.host_buffer_bytes(1, 2, 2, 128, 128, 64)
    buf = torch.empty(need - 1, dtype=torch.uint8, device="cuda")
    with pytest.raises(_lib.AttnError) as e:
        _lib.attn_fwd_host(q, k, v, causal=True, device_buffer=buf)
    assert e.value.status == _lib.ATTN_ERR_WORKSPACE


def test_host_entry_asynchronous_on_a_stream():
    """Enqueued on a side stream without synchronising: the outputs are
    complete once that stream is."""
    q, k, v = (t.pin_memory() for t in make_qkv(2, 3, 200, 700, 64, BF16, seed=73))
    s = torch.cuda.Stream()
    o = torch.full(q.shape, float("nan"), dtype=q.dtype).pin_memory()
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32).pin_memory()
    _lib.attn_fwd_host(q, k, v, causal=True, out=o, lse=lse, stream=s, synchronize=False)
    s.synchronize()
    compare(o.double().numpy(), lse.double().numpy(), oracle_fwd(q, k, v, True), BF16,
            "host entry, side stream")
    assert not np.isnan(o.double().numpy()).any()


LARGE_CASES = [
    # B, h_q, h_kv, T_q, T_kv, d, dtype, causal: large inputs, enqueued on a
    # side stream
    (4, 8, 8, 1, 16384, 128, BF16, False),    # decode, 256 MiB in
    (1, 8, 2, 64, 33000, 128, F16, True),     # grouped-query prefill, ~32 MiB in
]


@pytest.mark.parametrize("case", LARGE_CASES, ids=lambda c: "x".join(str(int(x)) for x in c))
def test_host_entry_large_inputs(case):
    """Large pinned inputs on a side stream, nothing synchronised before that
    stream is: the result matches the oracle and, bit for bit, the
    device-pointer path."""
    B, hq, hkv, tq, tk, d, dt, causal = case
    q, k, v = (t.pin_memory() for t in make_qkv(B, hq, tq, tk, d, dt, seed=74, h_kv=hkv))
    s = torch.cuda.Stream()
    o = torch.full(q.shape, float("nan"), dtype=q.dtype).pin_memory()
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32).pin_memory()
    _lib.attn_fwd_host(q, k, v, causal=causal, out=o, lse=lse, stream=s, synchronize=False)
    s.synchronize()
    st, word = _lib.get_device_error()
    assert st == _lib.ATTN_OK, f"device status {st} word {word:#x}"
    ref = oracle_fwd(q, k, v, causal) if hq == hkv else oracle_fwd_gqa(q, k, v, causal)
    compare(o.double().numpy(), lse.double().numpy(), ref, dt, f"host entry large {case}")
    o_dev, lse_dev = _device_ref(q, k, v, causal)
    assert torch.equal(o, o_dev) and torch.equal(lse, lse_dev)
