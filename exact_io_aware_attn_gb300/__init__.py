"""Exact IO-aware attention forward for GB300 (sm_103a).

The compute path is the C-ABI library libattn.so (hand-written CUDA kernels
under csrc/, declared in include/attn.h: forward prefill and decode, grouped-
query attention, and the backward pass); this package is its thin ctypes
binding plus the seeded input generator and the work counter the benchmark
uses. Importing the package does not load the library; the first call does,
and fails loudly if it has not been built.
"""

from ._lib import (  # noqa: F401
    AttnError,
    abi_version,
    bwd_workspace_bytes,
    attn_bwd,
    attn_fwd,
    attn_fwd_decode_noalloc,
    attn_fwd_gqa,
    attn_fwd_host,
    attn_fwd_naive,
    attn_fwd_paged_decode,
    attn_fwd_splitkv,
    decode_num_splits,
    fwd_raw,
    get_device_error,
    gqa_workspace_bytes,
    host_buffer_bytes,
    last_kernel_name,
    naive_workspace_bytes,
    paged_workspace_bytes,
    splitkv_workspace_bytes,
    status_string,
    workspace_bytes,
)
