"""Planted mistakes in copies of the oracle must each fail a pin.

This shows that the pins in oracle_pins.py are strong enough: a dropped
rescale, a wrong sign, an off-by-one mask, a transposed operand, a missing
normalisation or a wrong default scale in the oracle would not go unnoticed.
Mutants are built here on the CPU; the real oracle is never modified.
"""

import math
import types

import numpy as np
import pytest

import oracle
from oracle_pins import real_oracle, run_all


def _with(**over):
    base = vars(real_oracle()).copy()
    base.update(over)
    ns = types.SimpleNamespace(**base)
    if "standard_attention" in over and "standard_attention_row" not in over:
        def row(q, k, v, scale=None, _f=over["standard_attention"]):
            o, l = _f(np.asarray(q, dtype=np.float64)[None, :], k, v, scale=scale)
            return o[0], float(l[0])
        ns.standard_attention_row = row
    return ns


def _std_factory(mask_fn=None, lse_fn=None, transpose_k=False, normalise=True,
                 default_scale=lambda d: 1.0 / math.sqrt(d), rows_relative=False):
    def std(q, k, v, scale=None, causal=False, rows=None):
        q = np.asarray(q, dtype=np.float64)
        k = np.asarray(k, dtype=np.float64)
        v = np.asarray(v, dtype=np.float64)
        t_q, t_kv, d = q.shape[-2], k.shape[-2], q.shape[-1]
        if scale is None:
            scale = default_scale(d)
        lead = q.shape[:-2]
        rws = np.arange(t_q) if rows is None else np.asarray(rows)
        out = np.empty(lead + (len(rws), v.shape[-1]))
        lse = np.empty(lead + (len(rws),))
        for idx in np.ndindex(*lead):
            kk = k[idx]
            s = scale * (q[idx][rws] @ (kk if transpose_k else kk.T))
            if causal:
                # a selected row's causal position: its absolute index (or,
                # planted, its position among the selected rows)
                pos = np.arange(len(rws)) if rows_relative else rws
                vis = (mask_fn or (lambda i, j, off: j <= i + off))(
                    pos[:, None], np.arange(t_kv)[None, :], t_kv - t_q)
                s = np.where(vis, s, -np.inf)
            m = s.max(axis=1, keepdims=True)
            p = np.exp(s - m)
            l = p.sum(axis=1, keepdims=True)
            o = p @ v[idx]
            out[idx] = o / l if normalise else o
            lse[idx] = (lse_fn or (lambda m, l: m + np.log(l)))(m, l)[:, 0]
        return out, lse
    return std


def _online_factory(rescale=True, sign=1.0):
    def online(q, k, v, block, scale=None, return_state=False):
        q = np.asarray(q, dtype=np.float64)
        if scale is None:
            scale = 1.0 / math.sqrt(q.shape[0])
        m, l, o = -np.inf, 0.0, np.zeros(v.shape[1])
        for st in range(0, k.shape[0], block):
            s = scale * (k[st:st + block] @ q)
            m_new = max(m, float(s.max()))
            alpha = math.exp(sign * (m - m_new)) if rescale else 1.0
            p = np.exp(s - m_new)
            l = l * alpha + p.sum()
            o = o * alpha + p @ v[st:st + block]
            m = m_new
        return o / l
    return online


def _states_no_rescale(scores, block):
    s = np.asarray(scores, dtype=np.float64)
    m, l, out = -np.inf, 0.0, []
    for st in range(0, len(s), block):
        sb = s[st:st + block]
        m = max(m, float(sb.max()))
        l = l + float(np.exp(sb - m).sum())
        out.append((m, l))
    return out


def _merge_unweighted(ms, ls, os_):
    ms, ls, os_ = (np.asarray(x, dtype=np.float64) for x in (ms, ls, os_))
    o = os_.sum(axis=0) / ls.sum()
    return o, float(ms.max() + math.log(ls.sum()))


def _gqa_modulo_mapping(q, k, v, scale=None, causal=False, rows=None):
    # planted mistake: query head i uses key/value head i % h_kv
    h_q, h_kv = q.shape[1], k.shape[1]
    outs, lses = [], []
    for i in range(h_q):
        o, l = oracle.standard_attention(q[:, i], k[:, i % h_kv], v[:, i % h_kv], scale=scale,
                                         causal=causal, rows=rows)
        outs.append(o)
        lses.append(l)
    return np.stack(outs, axis=1), np.stack(lses, axis=1)


def _split_kv_with(merge):
    def f(q, k, v, num_splits, scale=None):
        return merge(*oracle.split_partials(q, k, v, num_splits, scale=scale))
    return f


def _bwd_factory(drop_d=False, dk_from_ds=False, dq_scale=True, dv_unnormalised=False,
                 causal_off=0):
    def bwd(q, k, v, do, scale=None, causal=False):
        q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
        t_q, t_kv, d = q.shape[-2], k.shape[-2], q.shape[-1]
        if scale is None:
            scale = 1.0 / math.sqrt(d)
        dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
        for idx in np.ndindex(*q.shape[:-2]):
            s_ = scale * (q[idx] @ k[idx].T)
            if causal:
                vis = np.arange(t_kv)[None, :] <= np.arange(t_q)[:, None] + (t_kv - t_q) + causal_off
                s_ = np.where(vis, s_, -np.inf)
            e = np.exp(s_ - s_.max(axis=1, keepdims=True))
            p = e / e.sum(axis=1, keepdims=True)
            dv[idx] = (e if dv_unnormalised else p).T @ do[idx]
            dp = do[idx] @ v[idx].T
            ds = p * dp if drop_d else p * (dp - (p * dp).sum(axis=1, keepdims=True))
            dq[idx] = (scale if dq_scale else 1.0) * (ds @ k[idx])
            # planted: dS (not its transpose) against Q, padded to the key count
            dk[idx] = scale * (ds.T @ q[idx] if not dk_from_ds else
                               np.resize(ds @ q[idx] if t_q == t_kv else ds.T @ q[idx][::-1],
                                         (t_kv, d)))
        return dq, dk, dv
    return bwd


def _gqa_bwd_overwrites(q, k, v, do, scale=None, causal=False):
    # planted mistake: each query head overwrites its key/value head's
    # gradient instead of adding to it
    q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
    group = q.shape[1] // k.shape[1]
    dq, dk, dv = np.empty_like(q), np.zeros_like(k), np.zeros_like(v)
    for i in range(q.shape[1]):
        j = i // group
        dq[:, i], dk[:, j], dv[:, j] = oracle.attention_backward(q[:, i], k[:, j], v[:, j], do[:, i],
                                                                 scale=scale, causal=causal)
    return dq, dk, dv


def _paged_factory(page_off=0, ignore_len=False, head_modulo=False):
    def paged(q, k_pages, v_pages, block_table, seq_lens, scale=None):
        q = np.asarray(q, dtype=np.float64)
        kp = np.asarray(k_pages, dtype=np.float64)
        vp = np.asarray(v_pages, dtype=np.float64)
        B, h_q, d = q.shape
        num_pages, h_kv, page_size, _ = kp.shape
        out = np.zeros((B, h_q, d))
        lse = np.full((B, h_q), -np.inf)
        for b in range(B):
            n = int(seq_lens[b]) if not ignore_len else block_table.shape[1] * page_size
            if n == 0:
                continue
            pages = [(int(p) + page_off) % num_pages for p in block_table[b, :-(-n // page_size)]]
            for i in range(h_q):
                j = (i % h_kv) if head_modulo else i // (h_q // h_kv)
                keys = np.concatenate([kp[p, j] for p in pages])[:n]
                vals = np.concatenate([vp[p, j] for p in pages])[:n]
                out[b, i], lse[b, i] = oracle.standard_attention_row(q[b, i], keys, vals, scale=scale)
        return out, lse
    return paged


MUTANTS = {
    "online_drops_rescale": _with(online_attention=_online_factory(rescale=False)),
    "online_rescale_wrong_sign": _with(online_attention=_online_factory(sign=-1.0)),
    "states_drop_rescale": _with(online_softmax_states=_states_no_rescale),
    "causal_excludes_diagonal": _with(standard_attention=_std_factory(
        mask_fn=lambda i, j, off: j < i + off)),
    "causal_top_left": _with(standard_attention=_std_factory(
        mask_fn=lambda i, j, off: j <= i)),
    "lse_drops_max": _with(standard_attention=_std_factory(lse_fn=lambda m, l: np.log(l))),
    "k_not_transposed": _with(standard_attention=_std_factory(transpose_k=True)),
    "output_not_normalised": _with(standard_attention=_std_factory(normalise=False)),
    "default_scale_1_over_d": _with(standard_attention=_std_factory(
        default_scale=lambda d: 1.0 / d)),
    "merge_ignores_weights": _with(split_kv_attention=_split_kv_with(_merge_unweighted)),
    "gqa_modulo_head_mapping": _with(gqa_attention=_gqa_modulo_mapping),
    "backward_drops_row_term": _with(attention_backward=_bwd_factory(drop_d=True)),
    "backward_dk_untransposed": _with(attention_backward=_bwd_factory(dk_from_ds=True)),
    "backward_dq_missing_scale": _with(attention_backward=_bwd_factory(dq_scale=False)),
    "backward_dv_unnormalised_p": _with(attention_backward=_bwd_factory(dv_unnormalised=True)),
    "backward_causal_excludes_diagonal": _with(attention_backward=_bwd_factory(causal_off=-1)),
    "gqa_backward_overwrites": _with(gqa_attention_backward=_gqa_bwd_overwrites),
    "rows_relative_causal_positions": _with(standard_attention=_std_factory(rows_relative=True)),
    "paged_off_by_one_page": _with(paged_decode_attention=_paged_factory(page_off=1)),
    "paged_ignores_length": _with(paged_decode_attention=_paged_factory(ignore_len=True)),
    "paged_modulo_head_mapping": _with(paged_decode_attention=_paged_factory(head_modulo=True)),
}


def test_real_oracle_passes_every_pin():
    assert run_all(real_oracle()) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    fails = run_all(MUTANTS[name])
    assert fails, f"planted mistake '{name}' passed every pin"
