"""The C-ABI library on any host (no GPU needed, no compute call made).

Checks that libattn.so builds, loads and exports every symbol include/attn.h
declares, and that every invalid argument is rejected with the right status
before anything is enqueued (validation runs before the first CUDA call, so
these calls are safe without a GPU).
"""

import ctypes
import os
import re

import pytest

from exact_io_aware_attn_gb300 import _lib, build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def L():
    build_mod.build()
    return _lib.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("attn_fwd", "attn_fwd_ex", "attn_workspace_bytes", "attn_get_device_error",
                 "attn_status_string", "attn_abi_version"):
        assert must in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), f"libattn.so does not export {name}"
        assert name in _lib.SIGNATURES, f"binding has no signature for {name}"


def test_binding_declares_nothing_extra():
    assert sorted(_lib.SIGNATURES) == declared_functions()


def test_abi_version_matches_header(L):
    m = re.search(r"#define ATTN_ABI_VERSION (\d+)", open(HEADER).read())
    assert L.attn_abi_version() == int(m.group(1))


def test_status_strings(L):
    for code, name in enumerate(["ATTN_OK", "ATTN_ERR_INVALID_ARG", "ATTN_ERR_UNSUPPORTED",
                                 "ATTN_ERR_CUDA", "ATTN_ERR_TIMEOUT", "ATTN_ERR_WORKSPACE"]):
        assert _lib.status_string(code) == name
    assert _lib.status_string(99) == "ATTN_ERR_UNKNOWN"


# fake, 16-byte aligned, non-overlapping addresses: validation never
# dereferences them
Q, K, V, O, LSE, WS = (0x100000 * i for i in range(1, 7))
GOOD = dict(B=2, h=3, T_q=100, T_kv=200, d=64, scale=0.125, causal=1, dtype=_lib.ATTN_BF16)


def call(**over):
    a = dict(GOOD)
    ptrs = dict(q=Q, k=K, v=V, o=O, lse=LSE)
    for key in list(over):
        if key in ptrs:
            ptrs[key] = over.pop(key)
    a.update(over)
    return _lib.fwd_raw(ptrs["q"], ptrs["k"], ptrs["v"], ptrs["o"], ptrs["lse"], a["B"], a["h"],
                        a["T_q"], a["T_kv"], a["d"], a["scale"], a["causal"], a["dtype"], None)


@pytest.mark.parametrize("over,status", [
    (dict(q=0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(k=0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(v=0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(o=0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(lse=0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(B=-1), _lib.ATTN_ERR_INVALID_ARG),
    (dict(h=-2), _lib.ATTN_ERR_INVALID_ARG),
    (dict(T_q=-1), _lib.ATTN_ERR_INVALID_ARG),
    (dict(T_kv=-1), _lib.ATTN_ERR_INVALID_ARG),
    (dict(T_kv=0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(d=0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(d=-64), _lib.ATTN_ERR_INVALID_ARG),
    (dict(d=96), _lib.ATTN_ERR_UNSUPPORTED),
    (dict(d=256), _lib.ATTN_ERR_UNSUPPORTED),
    (dict(d=32), _lib.ATTN_ERR_UNSUPPORTED),
    (dict(T_q=300, T_kv=200), _lib.ATTN_ERR_INVALID_ARG),      # causal needs T_q <= T_kv
    (dict(q=Q + 8), _lib.ATTN_ERR_INVALID_ARG),                 # misaligned
    (dict(k=K + 2), _lib.ATTN_ERR_INVALID_ARG),
    (dict(o=O + 4), _lib.ATTN_ERR_INVALID_ARG),
    (dict(lse=LSE + 2), _lib.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), _lib.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("inf")), _lib.ATTN_ERR_INVALID_ARG),
    (dict(scale=0.0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(scale=-0.125), _lib.ATTN_ERR_INVALID_ARG),
    (dict(dtype=2), _lib.ATTN_ERR_INVALID_ARG),
    (dict(dtype=-1), _lib.ATTN_ERR_INVALID_ARG),
    (dict(causal=2), _lib.ATTN_ERR_INVALID_ARG),
    (dict(o=Q), _lib.ATTN_ERR_INVALID_ARG),                     # output aliases an input
    (dict(o=K + 64), _lib.ATTN_ERR_INVALID_ARG),                # overlapping ranges
    (dict(lse=V), _lib.ATTN_ERR_INVALID_ARG),
    (dict(lse=O + 16), _lib.ATTN_ERR_INVALID_ARG),
    (dict(B=1 << 16, h=1 << 15), _lib.ATTN_ERR_UNSUPPORTED),    # B*h >= 2^31
])
def test_invalid_arguments_rejected_before_launch(L, over, status):
    assert call(**over) == status


@pytest.mark.parametrize("over", [dict(B=0), dict(h=0), dict(T_q=0),
                                  dict(B=0, q=0, k=0, v=0, o=0, lse=0),
                                  dict(T_q=0, T_kv=0, causal=0)])
def test_empty_problem_is_a_no_op(L, over):
    assert call(**over) == _lib.ATTN_OK
    assert _lib.last_kernel_name() == "none"


def _ex(num_splits, ws, nbytes, **over):
    a = dict(GOOD, T_q=1, causal=0)
    a.update(over)
    return _lib.fwd_raw(Q, K, V, O, LSE, a["B"], a["h"], a["T_q"], a["T_kv"], a["d"], a["scale"],
                        a["causal"], a["dtype"], None, num_splits, ws, nbytes)


def test_workspace_bytes_formula(L):
    B, h, T_kv = 32, 12, 16384
    for d in (64, 128):
        for s in (1, 16, 19, 64, 1024):
            assert _lib.workspace_bytes(B, h, 1, T_kv, d, s) == B * h * s * (d + 4) * 4
    # prefill needs no workspace; invalid sizes report 0
    assert _lib.workspace_bytes(B, h, 1024, 1024, 64, 0) == 0
    assert _lib.workspace_bytes(B, h, 1, T_kv, 96, 16) == 0
    assert _lib.workspace_bytes(B, h, 1, T_kv, 64, 1025) == 0
    assert _lib.workspace_bytes(-1, h, 1, T_kv, 64, 16) == 0


def test_auto_split_count_is_in_range(L):
    for (B, h, T) in ((32, 12, 16384), (1, 12, 16384), (1, 1, 100), (64, 12, 1024), (1, 1, 1)):
        s = _lib.decode_num_splits(B, h, T, 64)
        assert 1 <= s <= 1024
        assert s == 1 or T // s >= 128          # at least 128 keys per partition
        assert _lib.workspace_bytes(B, h, 1, T, 64, 0) == B * h * s * 68 * 4
    assert _lib.decode_num_splits(0, 12, 100, 64) == 0


@pytest.mark.parametrize("num_splits,ws,nbytes,status", [
    (-1, WS, 1 << 20, _lib.ATTN_ERR_INVALID_ARG),
    (1025, WS, 1 << 20, _lib.ATTN_ERR_INVALID_ARG),
    (16, 0, 1 << 20, _lib.ATTN_ERR_WORKSPACE),            # missing
    (16, WS, 100, _lib.ATTN_ERR_WORKSPACE),               # too small
    (16, WS + 4, 1 << 20, _lib.ATTN_ERR_WORKSPACE),       # misaligned
    (16, K, 1 << 20, _lib.ATTN_ERR_WORKSPACE),            # overlaps an input
])
def test_decode_workspace_errors(L, num_splits, ws, nbytes, status):
    assert _ex(num_splits, ws, nbytes) == status


def test_python_binding_rejects_cpu_tensors(L):
    import torch
    x = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        _lib.attn_fwd(x, x, x)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "libattn.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        _lib.lib()


def test_selftest_limit_validated_before_launch(L):
    assert _lib.selftest_wait_timeout(0) == _lib.ATTN_ERR_INVALID_ARG
    assert _lib.selftest_wait_timeout(2000001) == _lib.ATTN_ERR_INVALID_ARG


def _gqa(**over):
    a = dict(B=2, h_q=8, h_kv=2, T_q=1, T_kv=300, d=64, scale=0.125, causal=0,
             dtype=_lib.ATTN_BF16, num_splits=0)
    a.update(over)
    return _lib.fwd_gqa_raw(Q, K, V, O, LSE, a["B"], a["h_q"], a["h_kv"], a["T_q"], a["T_kv"],
                            a["d"], a["scale"], a["causal"], a["dtype"], a["num_splits"],
                            a.get("ws"), a.get("nbytes", 0), None)


@pytest.mark.parametrize("over,status", [
    (dict(h_kv=0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(h_kv=-1), _lib.ATTN_ERR_INVALID_ARG),
    (dict(h_kv=3), _lib.ATTN_ERR_INVALID_ARG),          # 8 is not a multiple of 3
    (dict(h_kv=16), _lib.ATTN_ERR_INVALID_ARG),         # more kv heads than query heads
    (dict(d=96), _lib.ATTN_ERR_UNSUPPORTED),
    (dict(num_splits=2000), _lib.ATTN_ERR_INVALID_ARG),
    (dict(ws=WS, nbytes=16), _lib.ATTN_ERR_WORKSPACE),  # caller workspace too small
    (dict(B=0), _lib.ATTN_OK),                          # empty
])
def test_gqa_arguments(L, over, status):
    assert _gqa(**over) == status


def test_gqa_workspace_bytes(L):
    assert _lib.gqa_workspace_bytes(2, 8, 2, 1, 300, 64, 16) == 2 * 8 * 16 * 68 * 4
    assert _lib.gqa_workspace_bytes(2, 8, 2, 300, 300, 64, 16) == 0     # prefill
    assert _lib.gqa_workspace_bytes(2, 8, 3, 1, 300, 64, 16) == 0       # invalid grouping
    assert _lib.gqa_workspace_bytes(2, 8, 8, 1, 300, 64, 0) == _lib.workspace_bytes(2, 8, 1, 300, 64, 0)


@pytest.mark.parametrize("h_q,h_kv", [(8, 2), (16, 2), (8, 4), (12, 12)])
@pytest.mark.parametrize("splits", [1, 16, 64, 65, 200, 1024])
def test_gqa_workspace_query_agrees_with_the_call(L, h_q, h_kv, splits):
    """The workspace query reports 0 exactly for the split counts the call
    rejects (on the tensor-core path, above 64; the rejection happens before
    any CUDA call), and the partials' size otherwise."""
    nbytes = _lib.gqa_workspace_bytes(2, h_q, h_kv, 1, 3000, 64, splits)
    if h_q // h_kv >= 4 and splits > 64:
        assert nbytes == 0
        # fake addresses 2^40 apart: no tensor overlaps another
        q, k, v, o, lse, ws = ((1 << 40) * i for i in range(1, 7))
        st = _lib.fwd_gqa_raw(q, k, v, o, lse, 2, h_q, h_kv, 1, 3000, 64, 0.125, 0,
                              _lib.ATTN_BF16, splits, ws, 1 << 30, None)
        assert st == _lib.ATTN_ERR_UNSUPPORTED
    else:
        assert nbytes == 2 * h_q * splits * 68 * 4


# backward: fake addresses for the extra tensors, spaced like the others
DO, DQ, DK, DV = (0x100000 * i for i in range(7, 11))


def _bwd(h_kv=None, **over):
    a = dict(GOOD)
    ptrs = dict(q=Q, k=K, v=V, o=O, do=DO, lse=LSE, dq=DQ, dk=DK, dv=DV)
    for key in list(over):
        if key in ptrs:
            ptrs[key] = over.pop(key)
    ws, nbytes = over.pop("ws", None), over.pop("nbytes", 0)
    a.update(over)
    return _lib.bwd_raw(ptrs["q"], ptrs["k"], ptrs["v"], ptrs["o"], ptrs["do"], ptrs["lse"],
                        ptrs["dq"], ptrs["dk"], ptrs["dv"], a["B"], a["h"],
                        a["h"] if h_kv is None else h_kv, a["T_q"], a["T_kv"], a["d"], a["scale"],
                        a["causal"], a["dtype"], ws, nbytes, None)


@pytest.mark.parametrize("over,status", [
    (dict(do=0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(dq=0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(dk=0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(dv=0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(q=0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(lse=0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(dq=DQ + 8), _lib.ATTN_ERR_INVALID_ARG),              # misaligned
    (dict(do=DO + 4), _lib.ATTN_ERR_INVALID_ARG),
    (dict(dq=Q), _lib.ATTN_ERR_INVALID_ARG),                   # gradient aliases an input
    (dict(dk=DO + 64), _lib.ATTN_ERR_INVALID_ARG),
    (dict(dv=LSE), _lib.ATTN_ERR_INVALID_ARG),
    (dict(dv=DK + 16), _lib.ATTN_ERR_INVALID_ARG),             # gradients overlap each other
    (dict(d=96), _lib.ATTN_ERR_UNSUPPORTED),
    (dict(T_q=300, T_kv=200), _lib.ATTN_ERR_INVALID_ARG),     # causal needs T_q <= T_kv
    (dict(scale=0.0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(dtype=3), _lib.ATTN_ERR_INVALID_ARG),
    (dict(ws=WS, nbytes=16), _lib.ATTN_ERR_WORKSPACE),         # too small
    (dict(ws=WS + 4, nbytes=1 << 20), _lib.ATTN_ERR_WORKSPACE),  # misaligned
    (dict(ws=DQ, nbytes=1 << 20), _lib.ATTN_ERR_WORKSPACE),    # overlaps a gradient
    (dict(ws=0, nbytes=1 << 20), _lib.ATTN_ERR_WORKSPACE),     # size without a buffer
    (dict(B=0), _lib.ATTN_OK),                                 # empty
    (dict(T_q=0), _lib.ATTN_OK),
])
def test_backward_arguments(L, over, status):
    assert _bwd(**over) == status


@pytest.mark.parametrize("h_kv,status", [(0, _lib.ATTN_ERR_INVALID_ARG),
                                         (2, _lib.ATTN_ERR_INVALID_ARG),   # 3 heads, 2 kv heads
                                         (6, _lib.ATTN_ERR_INVALID_ARG)])
def test_backward_gqa_grouping(L, h_kv, status):
    assert _bwd(h_kv=h_kv) == status


def test_backward_workspace_bytes(L):
    # two fp32 row terms per query row, rows padded to 128 per head
    assert _lib.bwd_workspace_bytes(2, 3, 100, 200, 64) == 2 * 2 * 3 * 128 * 4
    assert _lib.bwd_workspace_bytes(1, 1, 129, 129, 128) == 2 * 256 * 4
    assert _lib.bwd_workspace_bytes(1, 1, 100, 100, 96) == 0
    assert _lib.bwd_workspace_bytes(0, 1, 100, 100, 64) == 0


# paged decode: fake addresses for the pools and tables
KP, VP, TAB, LENS = (0x100000 * i for i in range(11, 15))


def _paged(**over):
    a = dict(B=2, h_q=4, h_kv=2, d=64, page_size=16, max_pages=8, num_pages=20, scale=0.125,
             dtype=_lib.ATTN_BF16, num_splits=0)
    ptrs = dict(q=Q, kp=KP, vp=VP, tab=TAB, lens=LENS, o=O, lse=LSE)
    for key in list(over):
        if key in ptrs:
            ptrs[key] = over.pop(key)
    ws, nbytes = over.pop("ws", None), over.pop("nbytes", 0)
    a.update(over)
    return _lib.paged_decode_raw(ptrs["q"], ptrs["kp"], ptrs["vp"], ptrs["tab"], ptrs["lens"],
                                 ptrs["o"], ptrs["lse"], a["B"], a["h_q"], a["h_kv"], a["d"],
                                 a["page_size"], a["max_pages"], a["num_pages"], a["scale"],
                                 a["dtype"], a["num_splits"], ws, nbytes, None)


@pytest.mark.parametrize("over,status", [
    (dict(q=0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(kp=0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(tab=0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(lens=0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(kp=KP + 8), _lib.ATTN_ERR_INVALID_ARG),          # misaligned pool
    (dict(tab=TAB + 2), _lib.ATTN_ERR_INVALID_ARG),        # misaligned table
    (dict(page_size=0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(page_size=24), _lib.ATTN_ERR_INVALID_ARG),       # not a power of two
    (dict(page_size=1 << 17), _lib.ATTN_ERR_INVALID_ARG),
    (dict(max_pages=0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(num_pages=0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(h_kv=3), _lib.ATTN_ERR_INVALID_ARG),             # 4 heads not a multiple of 3
    (dict(h_kv=0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(d=96), _lib.ATTN_ERR_UNSUPPORTED),
    (dict(num_splits=1025), _lib.ATTN_ERR_INVALID_ARG),
    (dict(o=KP + 64), _lib.ATTN_ERR_INVALID_ARG),          # output overlaps the pool
    (dict(lse=TAB), _lib.ATTN_ERR_INVALID_ARG),            # lse overlaps the table
    (dict(ws=WS, nbytes=16, num_splits=8), _lib.ATTN_ERR_WORKSPACE),
    (dict(ws=LENS, nbytes=1 << 20, num_splits=8), _lib.ATTN_ERR_WORKSPACE),
    (dict(page_size=65536, max_pages=1 << 16), _lib.ATTN_ERR_UNSUPPORTED),
    (dict(B=0), _lib.ATTN_OK),
])
def test_paged_decode_arguments(L, over, status):
    assert _paged(**over) == status


def test_paged_workspace_bytes(L):
    assert _lib.paged_workspace_bytes(2, 4, 2, 64, 16, 8, 5) == 2 * 4 * 5 * 68 * 4
    assert _lib.paged_workspace_bytes(2, 4, 4, 128, 16, 8, 3) == 2 * 4 * 3 * 132 * 4
    assert _lib.paged_workspace_bytes(2, 8, 2, 64, 16, 8, 5) == 2 * 8 * 5 * 68 * 4   # tensor cores
    assert _lib.paged_workspace_bytes(2, 8, 2, 64, 16, 8, 1) == 0   # one partition: none
    assert _lib.paged_workspace_bytes(2, 4, 2, 64, 24, 8, 5) == 0
    assert _lib.paged_workspace_bytes(2, 4, 3, 64, 16, 8, 5) == 0
    assert _lib.paged_workspace_bytes(0, 4, 2, 64, 16, 8, 5) == 0


def _splitkv(**over):
    a = dict(B=1, h_q=4, h_kv=2, T_q=256, T_kv=4096, d=64, scale=0.125, causal=1,
             dtype=_lib.ATTN_BF16, num_splits=8)
    ws, nbytes = over.pop("ws", None), over.pop("nbytes", 0)
    a.update(over)
    return _lib.splitkv_raw(Q, K, V, O, LSE, a["B"], a["h_q"], a["h_kv"], a["T_q"], a["T_kv"],
                            a["d"], a["scale"], a["causal"], a["dtype"], a["num_splits"], ws,
                            nbytes, None)


@pytest.mark.parametrize("over,status", [
    (dict(T_q=1), _lib.ATTN_ERR_INVALID_ARG),            # one row: the decode path
    (dict(num_splits=65), _lib.ATTN_ERR_INVALID_ARG),
    (dict(num_splits=-1), _lib.ATTN_ERR_INVALID_ARG),
    (dict(h_kv=3), _lib.ATTN_ERR_INVALID_ARG),
    (dict(d=96), _lib.ATTN_ERR_UNSUPPORTED),
    (dict(T_q=5000, T_kv=4096), _lib.ATTN_ERR_INVALID_ARG),   # causal needs T_q <= T_kv
    (dict(ws=WS, nbytes=64), _lib.ATTN_ERR_WORKSPACE),   # too small for 8 partitions
    (dict(ws=Q, nbytes=1 << 30), _lib.ATTN_ERR_WORKSPACE),  # overlaps q
    (dict(B=0), _lib.ATTN_OK),
])
def test_splitkv_arguments(L, over, status):
    assert _splitkv(**over) == status


def test_splitkv_workspace_bytes(L):
    assert _lib.splitkv_workspace_bytes(1, 4, 256, 4096, 64, 8) == 4 * 256 * 8 * 68 * 4
    assert _lib.splitkv_workspace_bytes(1, 4, 256, 4096, 64, 1) == 0
    assert _lib.splitkv_workspace_bytes(1, 4, 1, 4096, 64, 8) == 0


def _host(**over):
    a = dict(B=1, h_q=4, h_kv=2, T_q=256, T_kv=1024, d=64, scale=0.125, causal=1,
             dtype=_lib.ATTN_BF16)
    buf, nbytes = over.pop("buf", WS), over.pop("nbytes", 64)
    a.update(over)
    return _lib.fwd_host_raw(Q, K, V, O, LSE, a["B"], a["h_q"], a["h_kv"], a["T_q"], a["T_kv"],
                             a["d"], a["scale"], a["causal"], a["dtype"], buf, nbytes, None)


@pytest.mark.parametrize("over,status", [
    (dict(h_kv=0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(h_kv=3), _lib.ATTN_ERR_INVALID_ARG),
    (dict(d=96), _lib.ATTN_ERR_UNSUPPORTED),
    (dict(dtype=7), _lib.ATTN_ERR_INVALID_ARG),
    (dict(T_q=2000), _lib.ATTN_ERR_INVALID_ARG),          # causal needs T_q <= T_kv
    (dict(), _lib.ATTN_ERR_WORKSPACE),                    # 64 bytes: far too small
    (dict(buf=None, nbytes=1 << 30), _lib.ATTN_ERR_WORKSPACE),
    (dict(buf=WS + 8, nbytes=1 << 30), _lib.ATTN_ERR_WORKSPACE),  # misaligned
    (dict(B=0), _lib.ATTN_OK),
])
def test_host_entry_arguments(L, over, status):
    """attn_fwd_host checks its host pointers and the device buffer before
    the first copy is enqueued."""
    assert _host(**over) == status


def test_host_buffer_bytes(L):
    # q, k, v, o, lse each at a 256-byte offset
    qo = 1 * 4 * 256 * 64 * 2
    kv = 1 * 2 * 1024 * 64 * 2
    ls = 1 * 4 * 256 * 4
    assert _lib.host_buffer_bytes(1, 4, 2, 256, 1024, 64) == 2 * qo + 2 * kv + ls
    assert _lib.host_buffer_bytes(1, 4, 2, 1, 1000, 128) == (
        2 * ((4 * 128 * 2 + 255) // 256 * 256) + 2 * (2 * 1000 * 128 * 2) + 256)
    assert _lib.host_buffer_bytes(1, 4, 3, 256, 1024, 64) == 0   # h_q not a multiple of h_kv
    assert _lib.host_buffer_bytes(0, 4, 2, 256, 1024, 64) == 0
    assert _lib.host_buffer_bytes(1, 4, 2, 256, 1024, 96) == 0


def test_host_binding_rejects_bad_tensors(L):
    """attn_fwd_host's wrapper checks shapes and dtypes before any library
    or CUDA call: 4-D contiguous CPU tensors of one 16-bit dtype."""
    import torch
    q = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        _lib.attn_fwd_host(q[0], q[0], q[0])                      # 3-D
    with pytest.raises(ValueError):
        _lib.attn_fwd_host(q, q.transpose(2, 3), q)                 # not contiguous
    with pytest.raises(TypeError):
        _lib.attn_fwd_host(q, q.to(torch.float16), q)               # mixed dtypes
    with pytest.raises(ValueError):
        _lib.attn_fwd_host(q, torch.zeros(1, 2, 8, 32, dtype=torch.bfloat16),
                           torch.zeros(1, 2, 8, 32, dtype=torch.bfloat16))  # d differs


def test_device_wrappers_reject_host_tensors(L):
    """Every wrapper that takes device tensors refuses CPU tensors with a
    TypeError before any library call (a host address handed to a kernel
    would fault)."""
    import torch
    x = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16)
    lse = torch.zeros(1, 2, 8, dtype=torch.float32)
    x1 = torch.zeros(1, 2, 1, 64, dtype=torch.bfloat16)
    pages = torch.zeros(4, 2, 16, 64, dtype=torch.bfloat16)
    table = torch.zeros(1, 4, dtype=torch.int32)
    lens = torch.ones(1, dtype=torch.int32)
    calls = [
        lambda: _lib.attn_fwd(x, x, x),
        lambda: _lib.attn_fwd_gqa(x, x, x),
        lambda: _lib.attn_fwd_splitkv(x, x, x),
        lambda: _lib.attn_bwd(x, x, x, x, lse, x),
        lambda: _lib.attn_fwd_decode_noalloc(x1, x, x, out=x1, lse=lse[:, :, :1]),
        lambda: _lib.attn_fwd_paged_decode(x1, pages, pages, table, lens),
    ]
    for call in calls:
        with pytest.raises(TypeError):
            call()


def test_host_binding_checks_outputs_and_buffer(L):
    """The shared checks on out and lse (shape, dtype, contiguity, kind of
    memory) and on the device buffer, through attn_fwd_host: all fail before
    any library call."""
    import torch
    q = torch.zeros(1, 4, 8, 64, dtype=torch.float16)
    kv = torch.zeros(1, 2, 16, 64, dtype=torch.float16)      # grouped-query: 2 key/value heads
    lse = torch.zeros(1, 4, 8, dtype=torch.float32)
    bad = [
        (dict(out=torch.zeros(1, 4, 8, 32, dtype=torch.float16), lse=lse), ValueError),  # shape
        (dict(out=torch.zeros(1, 4, 8, 64, dtype=torch.bfloat16), lse=lse), TypeError),  # dtype
        (dict(out=torch.zeros(1, 4, 64, 8, dtype=torch.float16).transpose(2, 3), lse=lse),
         ValueError),
        (dict(out=q.clone(), lse=torch.zeros(1, 4, 7)), ValueError),              # lse rows
        (dict(out=q.clone(), lse=torch.zeros(1, 4, 8, dtype=torch.float64)), TypeError),
        (dict(out=q.clone(), lse=torch.zeros(1, 8, 4).transpose(1, 2)), ValueError),
        (dict(out=q.clone(), lse=lse, device_buffer=torch.zeros(1024, dtype=torch.uint8)),
         TypeError),                                                             # not on a GPU
        (dict(out=q.clone(), lse=lse, device_buffer=b"\0" * 1024), TypeError),   # not a tensor
    ]
    for kwargs, exc in bad:
        with pytest.raises(exc):
            _lib.attn_fwd_host(q, kv, kv, **kwargs)
    with pytest.raises(ValueError):                                              # v unlike k
        _lib.attn_fwd_host(q, kv, torch.zeros(1, 2, 15, 64, dtype=torch.float16), out=q, lse=lse)
    with pytest.raises(TypeError):                                               # fp32 inputs
        _lib.attn_fwd_host(q.float(), kv.float(), kv.float(), out=q.float(), lse=lse)
    with pytest.raises(TypeError):
        _lib.attn_fwd_host([q], kv, kv, out=q, lse=lse)


def test_shared_checks_accept_valid_shapes():
    """The checks pass the layouts the wrappers document: grouped-query k/v,
    and (for the paged decode) q as [B, h_q, d] or [B, h_q, 1, d]."""
    import torch
    q = torch.zeros(2, 8, 5, 128, dtype=torch.bfloat16)
    kv = torch.zeros(2, 2, 9, 128, dtype=torch.bfloat16)
    assert _lib._check_qkv(q, kv, kv, cuda=False) == (2, 8, 2, 5, 9, 128)
    _lib._check_outputs(q, torch.empty_like(q), torch.zeros(2, 8, 5), (2, 8, 5), cuda=False)
    empty = torch.zeros(0, 8, 5, 128, dtype=torch.bfloat16)
    assert _lib._check_qkv(empty, kv[:0], kv[:0], cuda=False)[0] == 0


def test_fast_checks_accept_exactly_the_valid_calls():
    """_check_qkv and _check_outputs try the valid case in one expression
    and fall back to per-argument checks that raise. Over random argument
    sets (ranks, dtypes, shapes, strides, a tensor subclass), each accepts
    exactly the sets an independent statement of the rules accepts, and
    returns the sizes that statement gives."""
    import random

    import torch
    rng = random.Random(5)
    dtypes = [torch.bfloat16, torch.float16, torch.float32]

    def rand_tensor(shape, dtype):
        t = torch.zeros(shape, dtype=dtype)
        r = rng.random()
        if r < 0.1 and t.dim() >= 2 and t.shape[-1] > 1 and t.shape[-2] > 1:
            t = t.transpose(-1, -2)                          # strided view
        elif r < 0.15:
            t = torch.nn.Parameter(t, requires_grad=False)   # a Tensor subclass
        return t

    def shape4():
        return [rng.choice([1, 2]), rng.choice([1, 2, 4]), rng.choice([1, 3, 5]),
                rng.choice([64, 128])]

    accepted = rejected = 0
    for _ in range(3000):
        qs = shape4()
        ks = [qs[0], rng.choice([1, 2]), rng.choice([1, 7]), qs[3]]
        vs = list(ks)
        bad = rng.random()
        if bad < 0.1:
            ks[0] += 1
        elif bad < 0.2:
            vs[2] += 1
        elif bad < 0.25:
            qs = qs[:3]
        dq = rng.choice(dtypes) if rng.random() < 0.3 else torch.bfloat16
        dk = rng.choice(dtypes) if rng.random() < 0.1 else dq
        q, k, v = rand_tensor(qs, dq), rand_tensor(ks, dk), rand_tensor(vs, dq)
        ok = (q.dim() == 4 and k.dim() == 4 and q.dtype in (torch.bfloat16, torch.float16)
              and k.dtype == q.dtype and v.dtype == q.dtype and k.shape[0] == q.shape[0]
              and k.shape[3] == q.shape[3] and v.shape == k.shape
              and all(t.is_contiguous() for t in (q, k, v)))
        try:
            got = _lib._check_qkv(q, k, v, cuda=False)
        except (TypeError, ValueError):
            got = None
        assert (got is not None) == ok, (q.shape, q.dtype, k.shape, k.dtype, v.shape)
        if ok:
            assert got == (q.shape[0], q.shape[1], k.shape[1], q.shape[2], k.shape[2], q.shape[3])
            out = rand_tensor(list(q.shape) if rng.random() < 0.8 else [1, 1, 1, 1],
                              q.dtype if rng.random() < 0.9 else torch.float32)
            lse_shape = list(q.shape[:3]) if rng.random() < 0.8 else [q.shape[0], q.shape[1]]
            lse = rand_tensor(lse_shape, torch.float32 if rng.random() < 0.9 else torch.float64)
            ok_out = (out.shape == q.shape and out.dtype == q.dtype and out.is_contiguous()
                      and tuple(lse.shape) == tuple(q.shape[:3]) and lse.dtype == torch.float32
                      and lse.is_contiguous())
            try:
                _lib._check_outputs(q, out, lse, tuple(q.shape[:3]), cuda=False)
                fine = True
            except (TypeError, ValueError):
                fine = False
            assert fine == ok_out, (out.shape, out.dtype, lse.shape, lse.dtype)
            accepted += 1
        else:
            rejected += 1
    assert accepted > 500 and rejected > 500


def test_splitkv_workspace_bytes(L):
    """Split-KV prefill sizing: B*h*T_q*S*(d+4)*4 bytes for S partitions, 0
    for one partition or invalid sizes. The library's own choice (S = 0) keeps
    problems whose units fill half the SMs unsplit, and otherwise takes 2..64
    partitions of at least two 128-key tiles each."""
    assert _lib.splitkv_workspace_bytes(1, 8, 256, 16384, 128, 7) == 8 * 256 * 7 * 132 * 4
    assert _lib.splitkv_workspace_bytes(2, 3, 100, 300, 64, 4) == 6 * 100 * 4 * 68 * 4
    assert _lib.splitkv_workspace_bytes(1, 8, 256, 16384, 128, 1) == 0
    assert _lib.splitkv_workspace_bytes(1, 8, 256, 16384, 128, 65) == 0     # above 64
    assert _lib.splitkv_workspace_bytes(1, 8, 1, 16384, 128, 4) == 0        # one row: decode
    assert _lib.splitkv_workspace_bytes(1, 8, 256, 16384, 96, 4) == 0       # unsupported d
    assert _lib.splitkv_workspace_bytes(8, 12, 1024, 1024, 64, 0) == 0      # fills the device
    for (B, h, T_q, T_kv, d) in ((1, 8, 256, 16384, 128), (1, 1, 300, 8192, 64),
                                 (1, 2, 4096, 4096, 128), (2, 1, 200, 200, 64)):
        nbytes = _lib.splitkv_workspace_bytes(B, h, T_q, T_kv, d, 0)
        per_split = B * h * T_q * (d + 4) * 4
        assert nbytes % per_split == 0
        S = nbytes // per_split
        n_kv = -(-T_kv // 128)
        assert S == 0 or 2 <= S <= min(64, n_kv // 2), (B, h, T_q, T_kv, d, S)
    # a long context behind a few query rows is split
    assert _lib.splitkv_workspace_bytes(1, 8, 256, 16384, 128, 0) > 0
