"""The element-wise parity gate against a model of the forward's rounding (no GPU).

The GPU parity tests hold every output element to a gate derived from the
arithmetic (parity_helpers.compare): fp32 accumulation, P rounded once to the
16-bit input type before the PV product (its row sum l taken from the
unrounded values), O rounded once at the end. This file runs a plain float32
model of exactly that rounding -- 128-key blocks, the lazy reference maximum
that moves only when a score exceeds it by 2^8, P rounded, O rounded -- and
checks, against the float64 oracle:

* on the workloads' input distributions and on inputs scaled by 3 (peaked
  rows, |O| up to ~12), the model's error stays inside the gate with margin,
  so the gate is not tighter than the arithmetic it describes;
* the same model with P rounded to two fewer mantissa bits (a 4x larger
  rounding step) breaks the gate on the scaled inputs, so the gate is tight
  enough to see such a change.

The model is not a second oracle: the GPU is always compared with the
float64 oracle, and this model only tests the gate.
"""

import math

import numpy as np
import pytest
import torch

from exact_io_aware_attn_gb300.inputs import BF16, F16, make_qkv
from parity_helpers import UNIT_ROUNDOFF, oracle_fwd, oracle_scale

TORCH_DT = {BF16: torch.bfloat16, F16: torch.float16}


def round_bits(p, bits):
    """Round to nearest with `bits` significant bits (a coarser 16-bit-like
    format; exponent range unlimited)."""
    m, e = torch.frexp(p)
    return torch.ldexp(torch.round(m * 2.0 ** bits) / 2.0 ** bits, e)


def rounding_model(q, k, v, causal, scale, dtype, p_bits=None, block=128, rebase=8.0):
    """O (float64 array) of the forward with the kernels' rounding, per head.
    q, k, v: CPU 16-bit tensors [B, h, T, d]."""
    B, h, T_q, d = q.shape
    T_kv = k.shape[2]
    sl2 = torch.tensor(scale * math.log2(math.e), dtype=torch.float32)
    out = np.empty((B, h, T_q, d))
    rows = torch.arange(T_q)[:, None]
    keys = torch.arange(T_kv)[None, :]
    visible = keys <= rows + (T_kv - T_q) if causal else torch.ones(T_q, T_kv, dtype=torch.bool)
    for b in range(B):
        for hh in range(h):
            qf, kf, vf = q[b, hh].float(), k[b, hh].float(), v[b, hh].float()
            s = torch.where(visible, qf @ kf.T, torch.tensor(-math.inf))
            m_used = torch.full((T_q,), -math.inf)
            l = torch.zeros(T_q)
            o = torch.zeros(T_q, d)
            for j0 in range(0, T_kv, block):
                sj = s[:, j0:j0 + block]
                m_tile = sj.max(dim=1).values * sl2
                move = m_tile > m_used + rebase
                alpha = torch.where(move & torch.isfinite(m_used), torch.exp2(m_used - m_tile),
                                    torch.where(move, torch.zeros(()), torch.ones(())))
                l = l * alpha
                o = o * alpha[:, None]
                m_used = torch.where(move, m_tile, m_used)
                m_ref = torch.where(torch.isfinite(m_used), m_used, torch.zeros(()))
                p = torch.exp2(sj * sl2 - m_ref[:, None])
                l = l + p.sum(dim=1)
                p16 = p.to(TORCH_DT[dtype]).float() if p_bits is None else round_bits(p, p_bits)
                o = o + p16 @ vf[j0:j0 + block]
            out[b, hh] = (o / l[:, None]).to(TORCH_DT[dtype]).double().numpy()
    return out


def gate_ratio(o, ref, dtype):
    o_ref, _, o_abs = ref
    u = UNIT_ROUNDOFF[dtype]
    bound = 1.25 * u * (o_abs + np.abs(o_ref)) + 1e-4
    return float((np.abs(o - o_ref) / bound).max())


CASES = [
    # B, h, T_q, T_kv, d, dtype, causal, input scale
    (1, 2, 256, 256, 64, F16, False, 1.0),
    (1, 2, 300, 300, 64, BF16, True, 1.0),
    (1, 1, 129, 500, 128, BF16, True, 1.0),
    (1, 2, 384, 384, 64, F16, True, 0.5),
    (1, 2, 300, 300, 64, BF16, True, 3.0),
    (1, 2, 256, 256, 64, F16, True, 3.0),
    (1, 1, 200, 700, 128, BF16, False, 3.0),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[2]}x{c[3]}_d{c[4]}_{'bf16' if c[5] else 'f16'}_"
                                                     f"{'causal' if c[6] else 'full'}_x{c[7]}")
def test_rounding_model_inside_the_gate(case):
    B, h, T_q, T_kv, d, dtype, causal, mult = case
    q, k, v = make_qkv(B, h, T_q, T_kv, d, dtype, mult, seed=11)
    scale = oracle_scale(d ** -0.5)
    ref = oracle_fwd(q, k, v, causal)
    ratio = gate_ratio(rounding_model(q, k, v, causal, scale, dtype), ref, dtype)
    assert ratio <= 0.9, f"the kernels' rounding reaches {ratio:.2f} of the gate"


@pytest.mark.parametrize("dtype", [BF16, F16])
def test_coarser_rounding_breaks_the_gate(dtype):
    """P rounded to two fewer significant bits than the 16-bit type (4x the
    rounding step) must be visible to the gate on peaked (x3) rows."""
    bits = 8 if dtype == BF16 else 11            # significant bits of the type
    worst = 0.0
    for seed in (11, 12):
        q, k, v = make_qkv(1, 2, 300, 300, 64, dtype, 3.0, seed=seed)
        ref = oracle_fwd(q, k, v, True)
        o = rounding_model(q, k, v, True, oracle_scale(0.125), dtype, p_bits=bits - 2)
        worst = max(worst, gate_ratio(o, ref, dtype))
    assert worst > 1.0, f"4x coarser rounding of P stays at {worst:.2f} of the gate"


@pytest.mark.parametrize("dtype,causal,pct", [(BF16, True, 3), (F16, True, 1), (BF16, False, 5),
                                               (F16, False, 1)])
def test_backward_gate_has_room_and_catches_a_small_dk_error(dtype, causal, pct):
    """The gradients' gate (parity_helpers.compare_grads): the oracle's own
    gradients rounded once to the 16-bit type pass with margin (about a
    quarter of the gate or less), and dK off by a few percent fails. The
    smallest caught error is 2% (bf16, causal), 3% (bf16, no mask) and 0.5%
    (fp16): dK is a cancelling sum (its rows of dS sum to zero), so bf16's
    gate leaves it more room."""
    from exact_io_aware_attn_gb300.inputs import make_dout
    from parity_helpers import compare_grads, oracle_bwd
    q, k, v = make_qkv(1, 2, 200, 200, 64, dtype, 1.0, seed=21)
    do = make_dout(1, 2, 200, 64, dtype, seed=21)
    ref = oracle_bwd(q, k, v, do, causal)
    rounded = [torch.from_numpy(g).to(TORCH_DT[dtype]).double().numpy() for g in ref[0]]
    assert compare_grads(rounded, ref, dtype, "oracle rounded") <= 0.5
    planted = [rounded[0], rounded[1] * (1 + pct / 100), rounded[2]]
    with pytest.raises(AssertionError, match="dk"):
        compare_grads(planted, ref, dtype, f"dK off by {pct}%")
