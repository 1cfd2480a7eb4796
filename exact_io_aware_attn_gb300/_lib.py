"""ctypes binding of libattn.so (the C ABI declared in include/attn.h).

Argument marshalling only: every step of the attention forward and backward
runs in the library's CUDA kernels. torch supplies device memory and the current
stream. There is no fallback: if the library is missing or a call fails,
an exception says so.
"""

from __future__ import annotations

import contextlib
import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libattn.so")

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_CUDA = 3
ATTN_ERR_TIMEOUT = 4
ATTN_ERR_WORKSPACE = 5
ATTN_F16 = 0
ATTN_BF16 = 1

# Every symbol include/attn.h declares, with its ctypes signature.
_VP, _I, _F, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "attn_fwd": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _F, _I, _I, _VP]),
    "attn_fwd_ex": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _F, _I, _I, _I, _VP, _SZ,
                         _VP]),
    "attn_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "attn_decode_num_splits": (_I, [_I, _I, _I, _I]),
    "attn_get_device_error": (_I, [_VP, ctypes.POINTER(ctypes.c_uint)]),
    "attn_status_string": (ctypes.c_char_p, [_I]),
    "attn_abi_version": (_I, []),
    "attn_last_kernel_name": (ctypes.c_char_p, []),
    "attn_fwd_decode_noalloc": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _F, _I, _I, _VP]),
    "attn_selftest_wait_timeout": (_I, [ctypes.c_uint, _VP]),
    "attn_fwd_gqa": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _F, _I, _I, _I, _VP,
                          _SZ, _VP]),
    "attn_gqa_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "attn_bwd": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _F, _I, _I,
                      _VP, _SZ, _VP]),
    "attn_bwd_gqa": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _F,
                          _I, _I, _VP, _SZ, _VP]),
    "attn_bwd_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "attn_fwd_paged_decode": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _I,
                                   _F, _I, _I, _VP, _SZ, _VP]),
    "attn_paged_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "attn_fwd_splitkv": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _F, _I, _I, _I, _VP,
                              _SZ, _VP]),
    "attn_splitkv_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "attn_fwd_host": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _F, _I, _I, _VP, _SZ,
                           _VP]),
    "attn_host_buffer_bytes": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "attn_fwd_naive": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _F, _I, _I, _VP, _SZ, _VP]),
    "attn_naive_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
}

# Bytes of the library-owned decode scratch behind attn_fwd_decode_noalloc.
NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})" if what else status_string(status))


def lib() -> ctypes.CDLL:
    """Load libattn.so (once). Raises if it has not been built."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"{LIB_PATH} is missing: build it with "
                        "`python -m exact_io_aware_attn_gb300.build` (there is no fallback path)")
                h = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in SIGNATURES.items():
                    fn = getattr(h, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = h
    return _lib


def status_string(status: int) -> str:
    return lib().attn_status_string(int(status)).decode()


def abi_version() -> int:
    return lib().attn_abi_version()


def last_kernel_name() -> str:
    return lib().attn_last_kernel_name().decode()


def workspace_bytes(B, h, T_q, T_kv, d, num_splits=0) -> int:
    return int(lib().attn_workspace_bytes(B, h, T_q, T_kv, d, num_splits))


def decode_num_splits(B, h, T_kv, d) -> int:
    return int(lib().attn_decode_num_splits(B, h, T_kv, d))


def get_device_error(stream=None):
    """Synchronise the stream, read and clear the device status word.
    Returns (status, recorded_word)."""
    word = ctypes.c_uint(0)
    st = lib().attn_get_device_error(_stream_ptr(stream), ctypes.byref(word))
    return int(st), int(word.value)


def gqa_workspace_bytes(B, h_q, h_kv, T_q, T_kv, d, num_splits=0) -> int:
    return int(lib().attn_gqa_workspace_bytes(B, h_q, h_kv, T_q, T_kv, d, num_splits))


def fwd_gqa_raw(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, h_q, h_kv, T_q, T_kv, d, scale, causal,
                dtype, num_splits=0, workspace_ptr=None, workspace_nbytes=0, stream_ptr=None) -> int:
    """Direct call of attn_fwd_gqa; returns the status code."""
    return int(lib().attn_fwd_gqa(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, h_q, h_kv, T_q, T_kv, d,
                                  float(scale), int(causal), int(dtype), int(num_splits),
                                  workspace_ptr, int(workspace_nbytes), stream_ptr))


def attn_fwd_gqa(q, k, v, *, scale=None, causal=False, out=None, lse=None, num_splits=0,
                 workspace=None, stream=None):
    """Grouped-query attention: q [B, h_q, T_q, d]; k, v [B, h_kv, T_kv, d]
    with h_q a multiple of h_kv. Returns (o like q, lse [B, h_q, T_q] fp32).
    The decode workspace is `workspace` (a CUDA tensor of at least
    gqa_workspace_bytes(...) bytes) or, when None, the library's
    stream-ordered allocation."""
    import torch
    B, h_q, h_kv, T_q, T_kv, d = _check_qkv(q, k, v)
    _same_device(q, k=k, v=v)
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, h_q, T_q), dtype=torch.float32, device=q.device)
    _check_outputs(q, out, lse, (B, h_q, T_q))
    wp, wn = _buffer("workspace", workspace, q.device)
    with torch.cuda.device(q.device):
        st = fwd_gqa_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                         B, h_q, h_kv, T_q, T_kv, d, scale, causal, _dtype_code(q), num_splits,
                         wp, wn, _stream_ptr(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_gqa")
    return out, lse


def selftest_wait_timeout(limit_us, stream=None) -> int:
    """Enqueue the failure-detection self-test (a bounded wait that runs
    out after limit_us); returns the status of the enqueue."""
    return int(lib().attn_selftest_wait_timeout(int(limit_us), _stream_ptr(stream)))


def _tensor(name, t, *, cuda=True, dim=None, shape=None, dtype=None):
    """Checks one tensor argument before anything reaches the library: the
    kind of memory (CUDA or CPU), rank, shape, dtype and contiguity. A wrong
    kind of tensor or dtype raises TypeError, the rest ValueError. The
    library reads raw addresses, so a tensor that is too small or strided
    would otherwise be read or written out of bounds."""
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.is_cuda is not cuda:
        raise TypeError(f"{name} must be a {'CUDA' if cuda else 'CPU'} tensor")
    if shape is not None:
        if t.shape != shape:
            raise ValueError(f"{name} must be shaped {tuple(shape)}, not {tuple(t.shape)}")
    elif dim is not None and t.dim() != dim:
        raise ValueError(f"{name} must have {dim} dimensions, not {t.dim()}")
    if dtype is not None and t.dtype is not dtype:
        raise TypeError(f"{name} must be {dtype}, not {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _same_device(q, **tensors):
    """Every CUDA tensor of one call lives on q's device (the library runs on
    the current device, which the wrappers set to q's)."""
    dev = q.get_device()
    for name, t in tensors.items():
        if t is not None and t.get_device() != dev:
            raise ValueError(f"{name} is on {t.device} but q on {q.device}: one device per call")


def _buffer(name, buf, device):
    """(address, bytes) of an optional caller buffer: a contiguous CUDA
    tensor on `device`, or (None, 0) when absent."""
    if buf is None:
        return None, 0
    _tensor(name, buf)
    if buf.device != device:
        raise ValueError(f"{name} is on {buf.device} but must be on {device}")
    return buf.data_ptr(), buf.numel() * buf.element_size()


def _check_qkv(q, k, v, *, cuda=True):
    """q [B, h_q, T_q, d]; k, v [B, h_kv, T_kv, d]; one 16-bit dtype.
    Returns (B, h_q, h_kv, T_q, T_kv, d)."""
    import torch
    T = torch.Tensor
    # the common, valid case in one expression (a few microseconds less per
    # call than the per-argument checks below, which name what is wrong)
    if (type(q) is T and type(k) is T and type(v) is T and q.is_cuda is cuda
            and k.is_cuda is cuda and v.is_cuda is cuda
            and (q.dtype is torch.bfloat16 or q.dtype is torch.float16)
            and k.dtype is q.dtype and v.dtype is q.dtype):
        qs, ks = q.shape, k.shape
        if (len(qs) == 4 and len(ks) == 4 and ks[0] == qs[0] and ks[3] == qs[3]
                and v.shape == ks and q.is_contiguous() and k.is_contiguous()
                and v.is_contiguous()):
            return qs[0], qs[1], ks[1], qs[2], ks[2], qs[3]
    _tensor("q", q, cuda=cuda, dim=4)
    _tensor("k", k, cuda=cuda, dim=4, dtype=q.dtype)
    B, h_q, T_q, d = q.shape
    Bk, h_kv, T_kv, dk = k.shape
    if Bk != B or dk != d:
        raise ValueError(f"k must be [B, h_kv, T_kv, d] with q's B = {B} and d = {d}, "
                         f"not {tuple(k.shape)}")
    _tensor("v", v, cuda=cuda, shape=k.shape, dtype=q.dtype)
    _dtype_code(q)
    return B, h_q, h_kv, T_q, T_kv, d


def _check_outputs(q, out, lse, lse_shape, *, cuda=True):
    """out like q (same shape and dtype), lse fp32 of lse_shape; both
    contiguous, on q's device when they are CUDA tensors."""
    import torch
    T = torch.Tensor
    if (type(out) is T and type(lse) is T and out.is_cuda is cuda and lse.is_cuda is cuda
            and out.dtype is q.dtype and lse.dtype is torch.float32 and out.shape == q.shape
            and lse.shape == lse_shape and out.is_contiguous() and lse.is_contiguous()
            and (not cuda or out.get_device() == lse.get_device() == q.get_device())):
        return
    _tensor("out", out, cuda=cuda, shape=q.shape, dtype=q.dtype)
    _tensor("lse", lse, cuda=cuda, shape=lse_shape, dtype=torch.float32)
    if cuda:
        _same_device(q, out=out, lse=lse)


def _stream_ptr(stream):
    if stream is None:
        import torch
        if not torch.cuda.is_available():
            return None
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def fwd_raw(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, h, T_q, T_kv, d, scale, causal, dtype,
            stream_ptr=None, num_splits=None, workspace_ptr=None, workspace_nbytes=0) -> int:
    """Direct call of attn_fwd (or attn_fwd_ex when num_splits is given) with
    raw addresses; returns the status code."""
    L = lib()
    if num_splits is None:
        return int(L.attn_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, h, T_q, T_kv, d,
                              float(scale), int(causal), int(dtype), stream_ptr))
    return int(L.attn_fwd_ex(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, h, T_q, T_kv, d,
                             float(scale), int(causal), int(dtype), int(num_splits),
                             workspace_ptr, int(workspace_nbytes), stream_ptr))


def fwd_decode_noalloc_raw(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, h, T_kv, d, scale, dtype,
                           num_splits=0, stream_ptr=None) -> int:
    """Direct call of attn_fwd_decode_noalloc; returns the status code."""
    return int(lib().attn_fwd_decode_noalloc(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, h, T_kv, d,
                                             float(scale), int(dtype), int(num_splits),
                                             stream_ptr))


def attn_fwd_decode_noalloc(q, k, v, *, out, lse, scale=None, num_splits=0, stream=None):
    """Decode (one query row per (b, h)) into caller-provided `out` and `lse`
    without allocating anything: for callers that cannot allocate device
    memory at call time. The partials live in a fixed library-owned device
    array (NOALLOC_SCRATCH_BYTES per device); calls that overlap on the GPU
    race on it. q: [B, h, 1, d]; k, v: [B, h, T_kv, d]; out like q; lse
    [B, h, 1] fp32."""
    import torch
    B, h, h_kv, T_q, T_kv, d = _check_qkv(q, k, v)
    if T_q != 1:
        raise ValueError("attn_fwd_decode_noalloc takes one query row per (b, h)")
    if h_kv != h:
        raise ValueError("attn_fwd_decode_noalloc takes one key/value head per query head")
    _same_device(q, k=k, v=v)
    _check_outputs(q, out, lse, (B, h, 1))
    if scale is None:
        scale = d ** -0.5
    # the library looks the scratch address up for the current device
    with torch.cuda.device(q.device):
        st = fwd_decode_noalloc_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                    lse.data_ptr(), B, h, T_kv, d, scale, _dtype_code(q),
                                    num_splits, _stream_ptr(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_decode_noalloc")
    return out, lse


def _dtype_code(t):
    import torch
    if t.dtype == torch.float16:
        return ATTN_F16
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    raise TypeError(f"unsupported dtype {t.dtype}: q, k, v must be float16 or bfloat16")


def attn_fwd(q, k, v, *, scale=None, causal=False, out=None, lse=None, num_splits=None,
             workspace=None, stream=None):
    """O, lse = softmax(scale * q k^T [+ causal mask]) v, on the GPU.

    q: [B, h, T_q, d]; k, v: [B, h, T_kv, d]; all contiguous CUDA tensors of
    one 16-bit dtype. Returns (o [B, h, T_q, d] same dtype, lse [B, h, T_q]
    fp32). `out`/`lse` may be preallocated. With `num_splits` (decode only)
    the call goes through attn_fwd_ex with a caller workspace (allocated here
    with torch if not given). Asynchronous on the current (or given) stream.
    """
    import torch
    B, h, h_kv, T_q, T_kv, d = _check_qkv(q, k, v)
    if h_kv != h:
        raise ValueError("k and v must have q's number of heads (attn_fwd_gqa takes fewer)")
    _same_device(q, k=k, v=v)
    dt = _dtype_code(q)
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, h, T_q), dtype=torch.float32, device=q.device)
    _check_outputs(q, out, lse, (B, h, T_q))
    with torch.cuda.device(q.device):
        sp = _stream_ptr(stream)          # q's device's current stream when none is given
        if num_splits is None:
            st = fwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                         B, h, T_q, T_kv, d, scale, causal, dt, sp)
        else:
            need = workspace_bytes(B, h, T_q, T_kv, d, num_splits)
            if workspace is None and need > 0:
                workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
            wp, wn = _buffer("workspace", workspace, q.device)
            st = fwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                         B, h, T_q, T_kv, d, scale, causal, dt, sp, num_splits, wp, wn)
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd")
    return out, lse


def bwd_workspace_bytes(B, h, T_q, T_kv, d) -> int:
    return int(lib().attn_bwd_workspace_bytes(B, h, T_q, T_kv, d))


def bwd_raw(q_ptr, k_ptr, v_ptr, o_ptr, do_ptr, lse_ptr, dq_ptr, dk_ptr, dv_ptr, B, h_q, h_kv,
            T_q, T_kv, d, scale, causal, dtype, workspace_ptr=None, workspace_nbytes=0,
            stream_ptr=None) -> int:
    """Direct call of attn_bwd (h_kv == h_q) or attn_bwd_gqa; returns the
    status code."""
    L = lib()
    if h_kv == h_q:
        return int(L.attn_bwd(q_ptr, k_ptr, v_ptr, o_ptr, do_ptr, lse_ptr, dq_ptr, dk_ptr, dv_ptr,
                              B, h_q, T_q, T_kv, d, float(scale), int(causal), int(dtype),
                              workspace_ptr, int(workspace_nbytes), stream_ptr))
    return int(L.attn_bwd_gqa(q_ptr, k_ptr, v_ptr, o_ptr, do_ptr, lse_ptr, dq_ptr, dk_ptr, dv_ptr,
                              B, h_q, h_kv, T_q, T_kv, d, float(scale), int(causal), int(dtype),
                              workspace_ptr, int(workspace_nbytes), stream_ptr))


def attn_bwd(q, k, v, o, lse, dout, *, scale=None, causal=False, dq=None, dk=None, dv=None,
             workspace=None, stream=None):
    """Gradients (dq, dk, dv) of attention from the forward's o and lse and
    dout = dL/dO. q, o, dout: [B, h_q, T_q, d]; k, v: [B, h_kv, T_kv, d]
    (h_kv < h_q: grouped-query attention); lse: fp32 [B, h_q, T_q] from the
    forward with the same scale and causal flag. The workspace is taken
    stream-ordered by the library unless given. Asynchronous."""
    import torch
    B, h_q, h_kv, T_q, T_kv, d = _check_qkv(q, k, v)
    _tensor("o", o, shape=q.shape, dtype=q.dtype)
    _tensor("dout", dout, shape=q.shape, dtype=q.dtype)
    _tensor("lse", lse, shape=(B, h_q, T_q), dtype=torch.float32)
    if scale is None:
        scale = d ** -0.5
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t, like in (("dq", dq, q), ("dk", dk, k), ("dv", dv, v)):
        _tensor(name, t, shape=like.shape, dtype=like.dtype)
    _same_device(q, k=k, v=v, o=o, dout=dout, lse=lse, dq=dq, dk=dk, dv=dv)
    wp, wn = _buffer("workspace", workspace, q.device)
    with torch.cuda.device(q.device):
        st = bwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
                     lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, h_q, h_kv,
                     T_q, T_kv, d, scale, causal, _dtype_code(q), wp, wn, _stream_ptr(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd")
    return dq, dk, dv


def paged_workspace_bytes(B, h_q, h_kv, d, page_size, max_pages_per_seq, num_splits=0) -> int:
    return int(lib().attn_paged_workspace_bytes(B, h_q, h_kv, d, page_size, max_pages_per_seq,
                                                num_splits))


def paged_decode_raw(q_ptr, kp_ptr, vp_ptr, table_ptr, lens_ptr, o_ptr, lse_ptr, B, h_q, h_kv, d,
                     page_size, max_pages, num_pages, scale, dtype, num_splits=0,
                     workspace_ptr=None, workspace_nbytes=0, stream_ptr=None) -> int:
    """Direct call of attn_fwd_paged_decode; returns the status code."""
    return int(lib().attn_fwd_paged_decode(q_ptr, kp_ptr, vp_ptr, table_ptr, lens_ptr, o_ptr,
                                           lse_ptr, B, h_q, h_kv, d, page_size, max_pages,
                                           num_pages, float(scale), int(dtype), int(num_splits),
                                           workspace_ptr, int(workspace_nbytes), stream_ptr))


def attn_fwd_paged_decode(q, k_pages, v_pages, block_table, seq_lens, *, scale=None, out=None,
                          lse=None, num_splits=0, workspace=None, stream=None):
    """Decode against a paged cache. q: [B, h_q, d] (or [B, h_q, 1, d]);
    k_pages, v_pages: [num_pages, h_kv, page_size, d]; block_table: int32
    [B, max_pages]; seq_lens: int32 [B]; all contiguous CUDA tensors.
    Returns (o like q, lse [B, h_q] fp32)."""
    import torch
    _tensor("q", q)
    if q.dim() not in (3, 4) or (q.dim() == 4 and q.shape[2] != 1):
        raise ValueError("q must be [B, h_q, d] or [B, h_q, 1, d]")
    _tensor("k_pages", k_pages, dim=4, dtype=q.dtype)
    num_pages, h_kv, page_size, d = k_pages.shape
    _tensor("v_pages", v_pages, shape=k_pages.shape, dtype=q.dtype)
    B, h_q = q.shape[0], q.shape[1]
    if q.shape[-1] != d:
        raise ValueError(f"q's last dimension must be the pages' d = {d}")
    _tensor("block_table", block_table, dim=2, dtype=torch.int32)
    if block_table.shape[0] != B:
        raise ValueError("block_table must be [B, max_pages]")
    _tensor("seq_lens", seq_lens, shape=(B,), dtype=torch.int32)
    _dtype_code(q)
    if scale is None:
        scale = d ** -0.5
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, h_q), dtype=torch.float32, device=q.device) if lse is None else lse
    _tensor("out", out, shape=q.shape, dtype=q.dtype)
    _tensor("lse", lse, dtype=torch.float32)
    if tuple(lse.shape) not in ((B, h_q), tuple(q.shape[:-1])):
        raise ValueError("lse must be [B, h_q] (or [B, h_q, 1] beside a [B, h_q, 1, d] q)")
    _same_device(q, k_pages=k_pages, v_pages=v_pages, block_table=block_table, seq_lens=seq_lens,
                 out=out, lse=lse)
    wp, wn = _buffer("workspace", workspace, q.device)
    with torch.cuda.device(q.device):
        st = paged_decode_raw(q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(),
                              block_table.data_ptr(), seq_lens.data_ptr(), out.data_ptr(),
                              lse.data_ptr(), B, h_q, h_kv, d, page_size, block_table.shape[1],
                              num_pages, scale, _dtype_code(q), num_splits, wp, wn,
                              _stream_ptr(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_paged_decode")
    return out, lse


def splitkv_workspace_bytes(B, h_q, T_q, T_kv, d, num_splits=0) -> int:
    return int(lib().attn_splitkv_workspace_bytes(B, h_q, T_q, T_kv, d, num_splits))


def splitkv_raw(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, h_q, h_kv, T_q, T_kv, d, scale, causal,
                dtype, num_splits=0, workspace_ptr=None, workspace_nbytes=0, stream_ptr=None) -> int:
    """Direct call of attn_fwd_splitkv; returns the status code."""
    return int(lib().attn_fwd_splitkv(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, h_q, h_kv, T_q, T_kv,
                                      d, float(scale), int(causal), int(dtype), int(num_splits),
                                      workspace_ptr, int(workspace_nbytes), stream_ptr))


def attn_fwd_splitkv(q, k, v, *, scale=None, causal=False, out=None, lse=None, num_splits=0,
                     workspace=None, stream=None):
    """Prefill (T_q >= 2) with the key range cut into num_splits partitions
    (0: the library's choice) and merged exactly. q [B, h_q, T_q, d]; k, v
    [B, h_kv, T_kv, d]. Returns (o like q, lse [B, h_q, T_q] fp32)."""
    import torch
    B, h_q, h_kv, T_q, T_kv, d = _check_qkv(q, k, v)
    _same_device(q, k=k, v=v)
    if scale is None:
        scale = d ** -0.5
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, h_q, T_q), dtype=torch.float32, device=q.device) if lse is None else lse
    _check_outputs(q, out, lse, (B, h_q, T_q))
    wp, wn = _buffer("workspace", workspace, q.device)
    with torch.cuda.device(q.device):
        st = splitkv_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                         B, h_q, h_kv, T_q, T_kv, d, scale, causal, _dtype_code(q), num_splits,
                         wp, wn, _stream_ptr(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_splitkv")
    return out, lse


def naive_workspace_bytes(B, h, T_q, T_kv) -> int:
    return int(lib().attn_naive_workspace_bytes(B, h, T_q, T_kv))


def naive_raw(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, h, T_q, T_kv, d, scale, causal, dtype,
              workspace_ptr=None, workspace_nbytes=0, stream_ptr=None) -> int:
    """Direct call of attn_fwd_naive; returns the status code."""
    return int(lib().attn_fwd_naive(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, h, T_q, T_kv, d,
                                    float(scale), int(causal), int(dtype), workspace_ptr,
                                    int(workspace_nbytes), stream_ptr))


def attn_fwd_naive(q, k, v, *, scale=None, causal=False, out=None, lse=None, workspace=None,
                   stream=None):
    """The materialising forward (S and P written to `workspace` as 16-bit
    [B, h, T_q, T_kv] matrices, then O = P V): the comparison baseline for
    the IO-aware kernels. q [B, h, T_q, d]; k, v [B, h, T_kv, d]. Returns (o
    like q, lse [B, h, T_q] fp32). `workspace`: a CUDA uint8 tensor of at
    least naive_workspace_bytes(...) bytes, else the stream-ordered
    allocator supplies it."""
    import torch
    B, h, h_kv, T_q, T_kv, d = _check_qkv(q, k, v)
    if h_kv != h:
        raise ValueError("attn_fwd_naive takes one key/value head per query head")
    _same_device(q, k=k, v=v)
    if scale is None:
        scale = d ** -0.5
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, h, T_q), dtype=torch.float32, device=q.device) if lse is None else lse
    _check_outputs(q, out, lse, (B, h, T_q))
    wp, wn = _buffer("workspace", workspace, q.device)
    with torch.cuda.device(q.device):
        st = naive_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                       B, h, T_q, T_kv, d, scale, causal, _dtype_code(q), wp, wn,
                       _stream_ptr(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_naive")
    return out, lse


def host_buffer_bytes(B, h_q, h_kv, T_q, T_kv, d) -> int:
    return int(lib().attn_host_buffer_bytes(B, h_q, h_kv, T_q, T_kv, d))


def fwd_host_raw(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, h_q, h_kv, T_q, T_kv, d, scale, causal,
                 dtype, buffer_ptr=None, buffer_nbytes=0, stream_ptr=None) -> int:
    """Direct call of attn_fwd_host (host addresses for q, k, v, o, lse);
    returns the status code."""
    return int(lib().attn_fwd_host(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, h_q, h_kv, T_q, T_kv, d,
                                   float(scale), int(causal), int(dtype), buffer_ptr,
                                   int(buffer_nbytes), stream_ptr))


def attn_fwd_host(q, k, v, *, scale=None, causal=False, out=None, lse=None, device_buffer=None,
                  stream=None, synchronize=True):
    """The forward on HOST tensors: q [B, h_q, T_q, d], k, v [B, h_kv, T_kv, d]
    (contiguous CPU tensors of one 16-bit dtype, ideally pinned). The library
    copies them to the GPU, runs the forward, and copies o and lse back into
    `out` / `lse` (CPU tensors; allocated pinned if not given). With
    synchronize=False the call only enqueues the work on the stream and the
    results are valid after it synchronises. `device_buffer` (a CUDA uint8
    tensor of at least host_buffer_bytes(...) bytes) holds the device copies;
    without it they come from the stream-ordered allocator."""
    import torch
    B, h_q, h_kv, T_q, T_kv, d = _check_qkv(q, k, v, cuda=False)
    dt = _dtype_code(q)
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    if lse is None:
        lse = torch.empty((B, h_q, T_q), dtype=torch.float32).pin_memory()
    _check_outputs(q, out, lse, (B, h_q, T_q), cuda=False)
    bp, bn, where = None, 0, contextlib.nullcontext()
    if device_buffer is not None:
        _tensor("device_buffer", device_buffer)
        bp, bn = device_buffer.data_ptr(), device_buffer.numel() * device_buffer.element_size()
        # the library works on the current device: make it the buffer's
        where = torch.cuda.device(device_buffer.device)
    with where:
        st = fwd_host_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                          lse.data_ptr(), B, h_q, h_kv, T_q, T_kv, d, scale, causal, dt, bp, bn,
                          _stream_ptr(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_host")
    if synchronize:
        if stream is None:
            torch.cuda.current_stream().synchronize()
        elif not isinstance(stream, int):
            stream.synchronize()
        else:
            torch.cuda.synchronize()
    return out, lse
