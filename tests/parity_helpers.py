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



# ---------------------------------------------------------------------------
# Backward pass
# ---------------------------------------------------------------------------
# Gate for the gradients, from the arithmetic of the kernels (all sums fp32):
#   dV_j = sum_i P_ij dO_i:  P rounded once to 16 bits (u P_ij) and dV
#        rounded once at the end (u |dV_j|);
#   dK_j = scale sum_i dS_ij Q_i and dQ_i = scale sum_j dS_ij K_j: dS rounded
#        once to 16 bits (u |dS_ij|); D_i = dO_i . o_i is formed from the
#        16-bit forward output o (u sum_c |dO_ic o_ic|, entering dS_ij times
#        P_ij); the result rounded once (u |X|).
# The fp32 sums over up to a few thousand terms add well under u for bf16
# and about u/2 for fp16, hence the factor 2. fp16 P and dS below the
# smallest normal (6.1e-5) keep an absolute precision of 2^-25, added as a
# term of its own.
BWD_FACTOR = 2.0


def gpu_bwd(q, k, v, do, causal, scale=None, workspace=None, o_lse=None):
    """Forward (for o and lse, unless given) then backward on the GPU.
    q, k, v, do: CPU 16-bit tensors. Returns float64 numpy (dq, dk, dv)."""
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    h_q, h_kv = q.shape[1], k.shape[1]
    if o_lse is None:
        if h_q == h_kv:
            o, lse = _lib.attn_fwd(qd, kd, vd, scale=scale, causal=causal)
        else:
            o, lse = _lib.attn_fwd_gqa(qd, kd, vd, scale=scale, causal=causal)
    else:
        o, lse = (t.to(dev) for t in o_lse)
    grads = [torch.full_like(t, float("nan")) for t in (qd, kd, vd)]   # unwritten shows up
    _lib.attn_bwd(qd, kd, vd, o, lse, dod, scale=scale, causal=causal, dq=grads[0], dk=grads[1],
                  dv=grads[2], workspace=workspace)
    torch.cuda.synchronize()
    st, word = _lib.get_device_error()
    assert st == _lib.ATTN_OK, f"device status {st} word {word:#x}"
    return tuple(g.double().cpu().numpy() for g in grads)


def oracle_bwd(q, k, v, do, causal, scale=None):
    """(dq, dk, dv) from the oracle, the magnitude terms the gate scales by u
    and the fp16 subnormal floor, all float64 numpy."""
    d = q.shape[-1]
    s = oracle_scale(d ** -0.5 if scale is None else scale)
    qn, kn, vn, dn = (t.double().numpy() for t in (q, k, v, do))
    B, h_q, T_q, _ = qn.shape
    h_kv = kn.shape[1]
    g = h_q // h_kv
    if h_q == h_kv:
        ref = oracle.attention_backward(qn, kn, vn, dn, scale=s, causal=causal)
    else:
        ref = oracle.gqa_attention_backward(qn, kn, vn, dn, scale=s, causal=causal)
    a_dq = np.zeros_like(qn)
    a_dk = np.zeros_like(kn)
    a_dv = np.zeros_like(vn)
    f_dq = np.zeros_like(qn)
    f_dk = np.zeros_like(kn)
    f_dv = np.zeros_like(vn)
    o_ref, _ = oracle.standard_attention(qn, np.repeat(kn, g, axis=1), np.repeat(vn, g, axis=1),
                                         scale=s, causal=causal)
    T_kv = kn.shape[2]
    vis = oracle.causal_visible(T_q, T_kv) if causal else np.ones((T_q, T_kv), dtype=bool)
    # fp16 values below the smallest normal keep an absolute precision of 2^-25
    sub = 2.0 ** -25 if q.dtype == torch.float16 else 0.0
    for b in range(B):
        for hq in range(h_q):
            hk = hq // g
            sc = s * (qn[b, hq] @ kn[b, hk].T)
            sc = np.where(vis, sc, -np.inf)
            e = np.exp(sc - sc.max(axis=1, keepdims=True))
            p = e / e.sum(axis=1, keepdims=True)
            dp = dn[b, hq] @ vn[b, hk].T
            ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
            r = (np.abs(dn[b, hq]) * np.abs(o_ref[b, hq])).sum(axis=1)   # sum_c |dO_ic o_ic|
            aq, ak, ado = np.abs(qn[b, hq]), np.abs(kn[b, hk]), np.abs(dn[b, hq])
            a_dv[b, hk] += p.T @ ado
            a_dk[b, hk] += s * (np.abs(ds).T @ aq + (p * r[:, None]).T @ aq)
            a_dq[b, hq] = s * (np.abs(ds) @ ak + r[:, None] * (p @ ak))
            f_dv[b, hk] += sub * (vis.T.astype(np.float64) @ ado)
            f_dk[b, hk] += s * sub * (vis.T.astype(np.float64) @ aq)
            f_dq[b, hq] = s * sub * (vis.astype(np.float64) @ ak)
    return ref, (a_dq, a_dk, a_dv), (f_dq, f_dk, f_dv)


def compare_grads(got, reference, dtype, what=""):
    """Element-wise gate on dq, dk, dv against oracle_bwd's output; returns
    the worst error/bound ratio."""
    ref, mag, floor = reference
    u = UNIT_ROUNDOFF[dtype]
    worst_ratio = 0.0
    for name, x, r, a, f in zip(("dq", "dk", "dv"), got, ref, mag, floor):
        assert np.isfinite(x).all(), f"{what}: {name} has non-finite (unwritten or NaN) elements"
        err = np.abs(x - r)
        bound = BWD_FACTOR * (u * (a + np.abs(r)) + f) + 1e-6
        ratio = err / bound
        i = int(np.argmax(ratio))
        assert ratio.flat[i] <= 1.0, (
            f"{what}: {name} element {np.unravel_index(i, x.shape)} = {x.flat[i]:.6g}, oracle "
            f"{r.flat[i]:.6g}, off by {err.flat[i]:.3e} > bound {bound.flat[i]:.3e}")
        worst_ratio = max(worst_ratio, float(ratio.flat[i]))
    return worst_ratio
