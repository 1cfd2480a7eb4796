"""Shared helpers for the GPU parity tests: run the CUDA path through the C
ABI, run the oracle on the very same 16-bit inputs, compare."""

from __future__ import annotations

import numpy as np
import torch

import oracle
from exact_io_aware_attn_gb300 import _lib
from exact_io_aware_attn_gb300.inputs import BF16, F16, make_qkv

# Tolerances the method states for 16-bit inputs with fp32 accumulation
# (N(0,1) workloads, |O| of order one).
O_TOL = 2e-2
LSE_TOL = 1e-3
# Element-wise gate derived from the arithmetic: P is rounded once to the
# 16-bit type before the PV product and O is rounded once at the end, each
# with unit roundoff u (2^-8 bf16, 2^-11 fp16); accumulation is fp32. The
# first rounding moves O_i by at most u * sum_j p_ij |v_jd| / l_i -- the
# attention-weighted mean of |V|, which the oracle computes by running on
# |V| -- and the second by u * |O_i|. The gate allows 1.25x that plus 1e-4.
UNIT_ROUNDOFF = {BF16: 2.0 ** -8, F16: 2.0 ** -11}


def oracle_scale(scale: float) -> float:
    """The float32 value the kernel receives, as float64."""
    return float(np.float32(scale))


def gpu_fwd(q, k, v, causal, scale=None, num_splits=None, check_status=True):
    """q, k, v: CPU 16-bit tensors. Returns (o float64 [B,h,T_q,d], lse float64)."""
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.full_like(qd, float("nan"))              # unwritten elements show up
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device=dev)
    _lib.attn_fwd(qd, kd, vd, scale=scale, causal=causal, out=o, lse=lse, num_splits=num_splits)
    torch.cuda.synchronize()
    if check_status:
        st, word = _lib.get_device_error()
        assert st == _lib.ATTN_OK, f"device status {st} word {word:#x}"
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


def oracle_fwd(q, k, v, causal, scale=None, rows=None):
    """(O, lse, O_abs): the oracle on (q, k, v), and O_abs = the oracle's
    output for |v| (the same weights applied to |V|)."""
    d = q.shape[-1]
    s = oracle_scale(d ** -0.5 if scale is None else scale)
    qn, kn, vn = q.double().numpy(), k.double().numpy(), v.double().numpy()
    o_ref, lse_ref = oracle.standard_attention(qn, kn, vn, scale=s, causal=causal, rows=rows)
    o_abs, _ = oracle.standard_attention(qn, kn, np.abs(vn), scale=s, causal=causal, rows=rows)
    return o_ref, lse_ref, o_abs


def compare(o, lse, ref, dtype, what="", absolute=True):
    """absolute=True also applies the fixed tolerances stated for the N(0,1)
    workloads; inputs scaled far beyond that (|O| up to ~12) are held to the
    rounding-derived gate alone."""
    o_ref, lse_ref, o_abs = ref
    assert np.isfinite(o).all(), f"{what}: non-finite output (unwritten or NaN)"
    assert np.isfinite(lse).all(), f"{what}: non-finite lse"
    err_o = np.abs(o - o_ref)
    err_l = np.abs(lse - lse_ref)
    if absolute:
        assert err_o.max() <= O_TOL, f"{what}: max|dO| = {err_o.max():.3e} > {O_TOL}"
    assert err_l.max() <= LSE_TOL, f"{what}: max|dlse| = {err_l.max():.3e} > {LSE_TOL}"
    u = UNIT_ROUNDOFF[dtype]
    bound = 1.25 * u * (o_abs + np.abs(o_ref)) + 1e-4
    worst = np.argmax(err_o / bound)
    assert (err_o <= bound).all(), (
        f"{what}: element {np.unravel_index(worst, o.shape)} off by "
        f"{err_o.flat[worst]:.3e} (bound {bound.flat[worst]:.3e})")
    return float(err_o.max()), float(err_l.max()), float(np.sqrt((err_o ** 2).mean()))


def check_case(B, h, T_q, T_kv, d, dtype, causal, mult=1.0, seed=0, scale=None, num_splits=None):
    q, k, v = make_qkv(B, h, T_q, T_kv, d, dtype, mult, seed)
    o, lse = gpu_fwd(q, k, v, causal, scale, num_splits)
    ref = oracle_fwd(q, k, v, causal, scale)
    return compare(o, lse, ref, dtype,
                   f"B{B} h{h} Tq{T_q} Tkv{T_kv} d{d} {'bf16' if dtype else 'f16'} causal={causal}",
                   absolute=mult <= 1.0)


def gpu_fwd_gqa(q, k, v, causal, num_splits=0):
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.full_like(qd, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device=dev)
    _lib.attn_fwd_gqa(qd, kd, vd, causal=causal, out=o, lse=lse, num_splits=num_splits)
    torch.cuda.synchronize()
    st, word = _lib.get_device_error()
    assert st == _lib.ATTN_OK, f"device status {st} word {word:#x}"
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


def oracle_fwd_gqa(q, k, v, causal, rows=None):
    s = oracle_scale(q.shape[-1] ** -0.5)
    qn, kn, vn = q.double().numpy(), k.double().numpy(), v.double().numpy()
    o_ref, lse_ref = oracle.gqa_attention(qn, kn, vn, scale=s, causal=causal, rows=rows)
    o_abs, _ = oracle.gqa_attention(qn, kn, np.abs(vn), scale=s, causal=causal, rows=rows)
    return o_ref, lse_ref, o_abs


def sample_rows(T_q, n_random=12, seed=0):
    """Rows that exercise every kind of tile position: first/last rows of
    tiles, the ragged tail, and a few random ones."""
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 63, 64, 127, 128, 129, 255, 256, T_q // 2, T_q - 129, T_q - 128, T_q - 2, T_q - 1]
    rows = [r for r in fixed if 0 <= r < T_q]
    rows += list(rng.integers(0, T_q, size=n_random))
    return np.unique(np.array(rows, dtype=np.int64))
