"""Pins for the oracle: checks against things other than the oracle itself.

Each check takes an implementation bundle (the real oracle, or a mutant with
a planted mistake) and returns a list of failure messages (empty = pinned).
The checks draw on:

* values the pages print (tests/golden/worked_example.json),
* a pure-Python brute force (no max subtraction, math.fsum) on tiny inputs,
* a library routine (torch scaled_dot_product_attention / logsumexp in
  float64 on the CPU),
* closed forms (one key, all-zero keys, causal row 0, one dominant key),
* invariants (key shift, joint key/value permutation, affine maps of V,
  folding a factor of q into the scale),
* exactness of the blocking and of the split merge (block sizes 1..n,
  partition counts 1..n+3),
* for the gradients: the library's autograd through float64
  scaled_dot_product_attention, central finite differences of the
  pure-Python brute force, closed forms (one key, equal value rows, causal
  row 0) and invariants (sum over keys of dK is zero, key shift, scale
  folding, linearity in dO).
"""

from __future__ import annotations

import json
import math
import os
import types

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def real_oracle():
    import oracle
    return types.SimpleNamespace(
        standard_attention=oracle.standard_attention,
        standard_attention_row=oracle.standard_attention_row,
        online_attention=oracle.online_attention,
        online_softmax_states=oracle.online_softmax_states,
        split_partials=oracle.split_partials,
        merge_partials=oracle.merge_partials,
        split_kv_attention=oracle.split_kv_attention,
        gqa_attention=oracle.gqa_attention,
        attention_backward=oracle.attention_backward,
        gqa_attention_backward=oracle.gqa_attention_backward,
        paged_decode_attention=oracle.paged_decode_attention,
    )


def _rng(seed):
    return np.random.default_rng(seed)


def _close(a, b, rtol=1e-12, atol=1e-12):
    return np.allclose(a, b, rtol=rtol, atol=atol)


# --------------------------------------------------------------------------
def check_worked_example(impl):
    with open(os.path.join(GOLDEN, "worked_example.json")) as f:
        ex = json.load(f)
    fails = []
    states = impl.online_softmax_states(ex["scores"], ex["block"])
    m1, l1 = states[0]
    if m1 != ex["after_block_1"]["m"]:
        fails.append(f"block-1 max {m1} != {ex['after_block_1']['m']}")
    if round(l1, ex["after_block_1"]["printed_decimals"]) != ex["after_block_1"]["l"]:
        fails.append(f"block-1 sum {l1:.6f} does not print as {ex['after_block_1']['l']}")
    m2, l2 = states[1]
    full_max = max(ex["scores"])
    full_sum = math.fsum(math.exp(s - full_max) for s in ex["scores"])
    if m2 != ex["after_block_2"]["m"] or m2 != full_max:
        fails.append(f"block-2 max {m2} != {full_max}")
    if not math.isclose(l2, full_sum, rel_tol=1e-14):
        fails.append(f"block-2 sum {l2!r} != full-row sum {full_sum!r}")
    return fails


def check_blockwise_equals_full(impl):
    fails = []
    rng = _rng(1)
    for n, d in ((1, 4), (7, 8), (33, 16)):
        for trial in range(2):
            q = rng.standard_normal(d) * 2.0
            k = rng.standard_normal((n, d)) * 2.0
            v = rng.standard_normal((n, d + 1))
            o_ref, _ = impl.standard_attention_row(q, k, v)
            for block in range(1, n + 2):
                o = impl.online_attention(q, k, v, block)
                if not _close(o, o_ref, rtol=1e-11, atol=1e-12):
                    fails.append(f"online(block={block}) != standard at n={n}")
                    break
    return fails


def _brute(q, k, v, scale, causal):
    """Pure-Python attention: weights exp(scale q.k) summed with fsum."""
    t_q, t_kv = len(q), len(k)
    out, lse = [], []
    for i in range(t_q):
        w = []
        for j in range(t_kv):
            if causal and j > i + (t_kv - t_q):
                w.append(0.0)
            else:
                dot = math.fsum(q[i][c] * k[j][c] for c in range(len(q[i])))
                w.append(math.exp(scale * dot))
        z = math.fsum(w)
        out.append([math.fsum(w[j] * v[j][c] for j in range(t_kv)) / z
                    for c in range(len(v[0]))])
        lse.append(math.log(z))
    return np.array(out), np.array(lse)


def check_bruteforce(impl):
    fails = []
    rng = _rng(2)
    for t_q, t_kv, d in ((1, 1, 3), (3, 5, 4), (5, 5, 4), (2, 8, 3), (8, 8, 5)):
        q = rng.standard_normal((t_q, d))
        k = rng.standard_normal((t_kv, d))
        v = rng.standard_normal((t_kv, d))
        for causal in (False, True):
            scale = 0.7
            o_b, l_b = _brute(q.tolist(), k.tolist(), v.tolist(), scale, causal)
            o, l = impl.standard_attention(q, k, v, scale=scale, causal=causal)
            if not (_close(o, o_b, rtol=1e-12, atol=1e-13)
                    and _close(l, l_b, rtol=1e-12, atol=1e-13)):
                fails.append(f"brute force mismatch t_q={t_q} t_kv={t_kv} causal={causal}")
    return fails


def check_library(impl):
    import torch
    import torch.nn.functional as F
    fails = []
    rng = _rng(3)
    for (b, h, t_q, t_kv, d) in ((1, 2, 16, 16, 8), (2, 1, 5, 19, 16), (1, 3, 1, 40, 8)):
        q = rng.standard_normal((b, h, t_q, d))
        k = rng.standard_normal((b, h, t_kv, d))
        v = rng.standard_normal((b, h, t_kv, d))
        tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
        for causal in (False, True):
            if causal:
                # bottom-right alignment, built independently of the oracle
                mask = torch.ones(t_q, t_kv, dtype=torch.bool).tril(diagonal=t_kv - t_q)
            else:
                mask = None
            o_lib = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask).numpy()
            s = (tq @ tk.transpose(-1, -2)) / math.sqrt(d)
            if mask is not None:
                s = s.masked_fill(~mask, float("-inf"))
            lse_lib = torch.logsumexp(s, dim=-1).numpy()
            o, lse = impl.standard_attention(q, k, v, causal=causal)
            if not (_close(o, o_lib, rtol=1e-10, atol=1e-12)
                    and _close(lse, lse_lib, rtol=1e-12, atol=1e-12)):
                fails.append(f"library mismatch shape={(b, h, t_q, t_kv, d)} causal={causal}")
    return fails


def check_closed_forms(impl):
    fails = []
    rng = _rng(4)
    d = 6
    # one key: O = V, lse = scale q.k
    q = rng.standard_normal((3, d))
    k = rng.standard_normal((1, d))
    v = rng.standard_normal((1, d))
    o, lse = impl.standard_attention(q, k, v, scale=0.5)
    if not (_close(o, np.repeat(v, 3, axis=0)) and _close(lse, 0.5 * (q @ k[0]))):
        fails.append("T_kv = 1 closed form")
    # all-zero keys: uniform weights, O = mean(V), lse = ln T_kv
    k0 = np.zeros((9, d))
    v9 = rng.standard_normal((9, d))
    o, lse = impl.standard_attention(q, k0, v9)
    if not (_close(o, np.repeat(v9.mean(axis=0, keepdims=True), 3, axis=0))
            and _close(lse, np.full(3, math.log(9)))):
        fails.append("K = 0 closed form")
    # causal, square: row 0 sees only key 0
    q5 = rng.standard_normal((5, d))
    k5 = rng.standard_normal((5, d))
    v5 = rng.standard_normal((5, d))
    o, lse = impl.standard_attention(q5, k5, v5, scale=0.3, causal=True)
    if not (_close(o[0], v5[0]) and math.isclose(lse[0], 0.3 * float(q5[0] @ k5[0]),
                                                  rel_tol=1e-12, abs_tol=1e-12)):
        fails.append("causal row 0 closed form")
    # causal, one query against a cache: sees every key (equals non-causal)
    o_c, l_c = impl.standard_attention(q5[:1], k5, v5, causal=True)
    o_n, l_n = impl.standard_attention(q5[:1], k5, v5, causal=False)
    if not (_close(o_c, o_n) and _close(l_c, l_n)):
        fails.append("one causal query must see the whole cache")
    # last causal row of a square problem sees every key
    o_l, _ = impl.standard_attention(q5[4:5], k5, v5, scale=0.3)
    if not _close(o[4], o_l[0]):
        fails.append("causal last row must equal the unmasked row")
    # one dominant key: weight -> 1
    kd = np.zeros((4, 2))
    kd[2] = [100.0, 0.0]
    qd = np.array([[10.0, 0.0]])
    vd = np.arange(8.0).reshape(4, 2)
    o, lse = impl.standard_attention(qd, kd, vd, scale=1.0)
    if not (_close(o[0], vd[2]) and math.isclose(lse[0], 1000.0, rel_tol=1e-12)):
        fails.append("dominant key closed form")
    return fails


def check_invariants(impl):
    fails = []
    rng = _rng(5)
    t_q, t_kv, d = 6, 11, 8
    q = rng.standard_normal((t_q, d))
    k = rng.standard_normal((t_kv, d))
    v = rng.standard_normal((t_kv, d))
    s = 0.4
    for causal in (False, True):
        o, lse = impl.standard_attention(q, k, v, scale=s, causal=causal)
        u = rng.standard_normal(d)
        o2, lse2 = impl.standard_attention(q, k + u, v, scale=s, causal=causal)
        if not (_close(o2, o, rtol=1e-10, atol=1e-11)
                and _close(lse2, lse + s * (q @ u), rtol=1e-10, atol=1e-11)):
            fails.append(f"key shift invariance (causal={causal})")
        a, b = -1.7, rng.standard_normal(d)
        o3, lse3 = impl.standard_attention(q, k, a * v + b, scale=s, causal=causal)
        if not (_close(o3, a * o + b, rtol=1e-10, atol=1e-11) and _close(lse3, lse)):
            fails.append(f"affine map of V (causal={causal})")
        o4, lse4 = impl.standard_attention(2.5 * q, k, v, scale=s / 2.5, causal=causal)
        if not (_close(o4, o, rtol=1e-10, atol=1e-11) and _close(lse4, lse, rtol=1e-10)):
            fails.append(f"scale folding (causal={causal})")
    perm = rng.permutation(t_kv)
    o, lse = impl.standard_attention(q, k, v, scale=s)
    o5, lse5 = impl.standard_attention(q, k[perm], v[perm], scale=s)
    if not (_close(o5, o, rtol=1e-10, atol=1e-11) and _close(lse5, lse, rtol=1e-12)):
        fails.append("joint key/value permutation")
    # rows= selects rows with absolute causal positions
    rows = np.array([5, 0, 3])
    o6, lse6 = impl.standard_attention(q, k, v, scale=s, causal=True, rows=rows)
    o7, lse7 = impl.standard_attention(q, k, v, scale=s, causal=True)
    if not (_close(o6, o7[rows]) and _close(lse6, lse7[rows])):
        fails.append("row selection must keep absolute causal positions")
    return fails


def check_split_merge(impl):
    fails = []
    rng = _rng(6)
    for n in (1, 5, 17):
        d = 8
        q = rng.standard_normal(d) * 2
        k = rng.standard_normal((n, d)) * 2
        v = rng.standard_normal((n, d))
        o_ref, lse_ref = impl.standard_attention_row(q, k, v)
        for splits in range(1, n + 4):
            o, lse = impl.split_kv_attention(q, k, v, splits)
            if not (_close(o, o_ref, rtol=1e-11, atol=1e-12)
                    and math.isclose(lse, lse_ref, rel_tol=1e-12, abs_tol=1e-12)):
                fails.append(f"split merge n={n} splits={splits}")
                break
    return fails


def check_gqa(impl):
    """Grouped-query attention against the library's float64 grouped SDPA,
    and its reductions: one query head per key/value head is standard
    attention; repeating each key/value head `group` times is the same."""
    import torch
    import torch.nn.functional as F
    fails = []
    rng = _rng(7)
    for (b, h_q, h_kv, t_q, t_kv, d) in ((2, 4, 2, 5, 9, 8), (1, 8, 2, 1, 33, 16), (1, 6, 3, 7, 7, 4)):
        q = rng.standard_normal((b, h_q, t_q, d))
        k = rng.standard_normal((b, h_kv, t_kv, d))
        v = rng.standard_normal((b, h_kv, t_kv, d))
        for causal in (False, True):
            if causal and t_q > t_kv:
                continue
            mask = (torch.ones(t_q, t_kv, dtype=torch.bool).tril(diagonal=t_kv - t_q)
                    if causal else None)
            o_lib = F.scaled_dot_product_attention(torch.from_numpy(q), torch.from_numpy(k),
                                                   torch.from_numpy(v), attn_mask=mask,
                                                   enable_gqa=True).numpy()
            o, lse = impl.gqa_attention(q, k, v, causal=causal)
            if not _close(o, o_lib, rtol=1e-10, atol=1e-12):
                fails.append(f"gqa vs library shape={(b, h_q, h_kv, t_q, t_kv, d)} causal={causal}")
            g = h_q // h_kv
            o_rep, lse_rep = impl.standard_attention(q, np.repeat(k, g, axis=1),
                                                     np.repeat(v, g, axis=1), causal=causal)
            if not (_close(o, o_rep) and _close(lse, lse_rep)):
                fails.append(f"gqa vs repeated heads shape={(b, h_q, h_kv)} causal={causal}")
    q = rng.standard_normal((1, 3, 4, 8))
    k = rng.standard_normal((1, 3, 6, 8))
    o1, l1 = impl.gqa_attention(q, k, k)
    o2, l2 = impl.standard_attention(q, k, k)
    if not (_close(o1, o2) and _close(l1, l2)):
        fails.append("gqa with one query head per key/value head must be standard attention")
    return fails


def _autograd_sdpa(q, k, v, do, causal, scale=None, gqa=False):
    """Gradients from the library: torch autograd through float64 SDPA."""
    import torch
    import torch.nn.functional as F
    tq, tk, tv = (torch.from_numpy(np.array(x)).requires_grad_(True) for x in (q, k, v))
    t_q, t_kv = q.shape[-2], k.shape[-2]
    mask = (torch.ones(t_q, t_kv, dtype=torch.bool).tril(diagonal=t_kv - t_q)
            if causal else None)
    o = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=scale, enable_gqa=gqa)
    o.backward(torch.from_numpy(np.array(do)))
    return tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


def check_backward_library(impl):
    fails = []
    rng = _rng(8)
    for (b, h, t_q, t_kv, d) in ((1, 2, 16, 16, 8), (2, 1, 5, 19, 16), (1, 3, 1, 40, 8),
                                 (1, 1, 7, 7, 4)):
        q = rng.standard_normal((b, h, t_q, d))
        k = rng.standard_normal((b, h, t_kv, d))
        v = rng.standard_normal((b, h, t_kv, d))
        do = rng.standard_normal((b, h, t_q, d))
        for causal in (False, True):
            for scale in (None, 0.3):
                ref = _autograd_sdpa(q, k, v, do, causal, scale)
                got = impl.attention_backward(q, k, v, do, scale=scale, causal=causal)
                for name, a, r in zip(("dq", "dk", "dv"), got, ref):
                    if not _close(a, r, rtol=1e-9, atol=1e-11):
                        fails.append(f"{name} vs library autograd shape={(b, h, t_q, t_kv, d)} "
                                     f"causal={causal} scale={scale}")
    return fails


def check_backward_finite_difference(impl):
    """Central differences of L = sum(O * dO), O from the pure-Python brute
    force, against the oracle's gradients on tiny inputs."""
    fails = []
    rng = _rng(9)
    eps = 1e-6
    for t_q, t_kv, d, causal in ((3, 4, 3, False), (3, 4, 3, True), (4, 4, 2, True)):
        q = rng.standard_normal((t_q, d))
        k = rng.standard_normal((t_kv, d))
        v = rng.standard_normal((t_kv, d))
        do = rng.standard_normal((t_q, d))
        scale = 0.6
        got = impl.attention_backward(q, k, v, do, scale=scale, causal=causal)

        def loss(qq, kk, vv):
            o, _ = _brute(qq.tolist(), kk.tolist(), vv.tolist(), scale, causal)
            return math.fsum((o * do).ravel().tolist())

        for which, (name, g) in enumerate(zip(("dq", "dk", "dv"), got)):
            x = [q, k, v][which]
            num = np.empty_like(x)
            for idx in np.ndindex(*x.shape):
                args_p = [q.copy(), k.copy(), v.copy()]
                args_m = [q.copy(), k.copy(), v.copy()]
                args_p[which][idx] += eps
                args_m[which][idx] -= eps
                num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            if not _close(g, num, rtol=1e-6, atol=1e-7):
                fails.append(f"{name} vs finite differences t_q={t_q} t_kv={t_kv} causal={causal}")
    return fails


def check_backward_closed_forms(impl):
    fails = []
    rng = _rng(10)
    d = 5
    # one key: P = 1 whatever the scores, so dQ = dK = 0 and dV = sum of dO
    q = rng.standard_normal((4, d))
    k1 = rng.standard_normal((1, d))
    v1 = rng.standard_normal((1, d))
    do = rng.standard_normal((4, d))
    dq, dk, dv = impl.attention_backward(q, k1, v1, do, scale=0.5)
    if not (_close(dq, 0 * dq) and _close(dk, 0 * dk) and _close(dv[0], do.sum(axis=0))):
        fails.append("T_kv = 1 gradients")
    # equal value rows: O = v whatever P is, so dQ = dK = 0; dV = P^T dO
    # still sums to the sum of dO over the keys (columns of P^T sum to 1)
    k6 = rng.standard_normal((6, d))
    v6 = np.repeat(rng.standard_normal((1, d)), 6, axis=0)
    for causal in (False, True):
        dq, dk, dv = impl.attention_backward(q, k6, v6, do, scale=0.5, causal=causal)
        if not (_close(dq, 0 * dq, atol=1e-12) and _close(dk, 0 * dk, atol=1e-12)
                and _close(dv.sum(axis=0), do.sum(axis=0))):
            fails.append(f"equal value rows gradients (causal={causal})")
    # causal, square: row 0 sees only key 0, so dQ[0] = 0 and dO[0] flows
    # into dV[0] alone
    q5 = rng.standard_normal((5, d))
    k5 = rng.standard_normal((5, d))
    v5 = rng.standard_normal((5, d))
    do5 = np.zeros((5, d))
    do5[0] = rng.standard_normal(d)
    dq, dk, dv = impl.attention_backward(q5, k5, v5, do5, scale=0.3, causal=True)
    if not (_close(dq[0], 0 * dq[0]) and _close(dv[0], do5[0]) and _close(dv[1:], 0 * dv[1:])
            and _close(dk, 0 * dk)):
        fails.append("causal row 0 gradients")
    # dO = 0: every gradient is 0
    dq, dk, dv = impl.attention_backward(q5, k5, v5, np.zeros((5, d)), causal=True)
    if not (_close(dq, 0 * dq) and _close(dk, 0 * dk) and _close(dv, 0 * dv)):
        fails.append("zero incoming gradient")
    return fails


def check_backward_invariants(impl):
    fails = []
    rng = _rng(11)
    t_q, t_kv, d = 6, 9, 4
    q = rng.standard_normal((t_q, d))
    k = rng.standard_normal((t_kv, d))
    v = rng.standard_normal((t_kv, d))
    do = rng.standard_normal((t_q, d))
    s = 0.45
    for causal in (False, True):
        dq, dk, dv = impl.attention_backward(q, k, v, do, scale=s, causal=causal)
        # rows of dS sum to zero, so the key gradients sum to zero
        if not _close(dk.sum(axis=0), np.zeros(d), atol=1e-12):
            fails.append(f"sum of dK over keys must vanish (causal={causal})")
        # a shift of every key leaves P, and so every gradient, unchanged
        u = rng.standard_normal(d)
        g2 = impl.attention_backward(q, k + u, v, do, scale=s, causal=causal)
        if not all(_close(a, b, rtol=1e-9, atol=1e-11) for a, b in zip(g2, (dq, dk, dv))):
            fails.append(f"key shift invariance of the gradients (causal={causal})")
        # folding a factor into q: dQ scales by 1/a, dK and dV do not change
        a = 2.5
        g3 = impl.attention_backward(a * q, k, v, do, scale=s / a, causal=causal)
        if not (_close(g3[0], dq / a, rtol=1e-9, atol=1e-11)
                and _close(g3[1], dk, rtol=1e-9, atol=1e-11) and _close(g3[2], dv)):
            fails.append(f"scale folding of the gradients (causal={causal})")
        # gradients are linear in dO
        g4 = impl.attention_backward(q, k, v, -3.0 * do, scale=s, causal=causal)
        if not all(_close(x4, -3.0 * x, rtol=1e-10, atol=1e-12) for x4, x in zip(g4, (dq, dk, dv))):
            fails.append(f"linearity in dO (causal={causal})")
    return fails


def check_backward_gqa(impl):
    fails = []
    rng = _rng(12)
    for (b, h_q, h_kv, t_q, t_kv, d) in ((2, 4, 2, 5, 9, 8), (1, 6, 3, 7, 7, 4)):
        q = rng.standard_normal((b, h_q, t_q, d))
        k = rng.standard_normal((b, h_kv, t_kv, d))
        v = rng.standard_normal((b, h_kv, t_kv, d))
        do = rng.standard_normal((b, h_q, t_q, d))
        for causal in (False, True):
            ref = _autograd_sdpa(q, k, v, do, causal, gqa=True)
            got = impl.gqa_attention_backward(q, k, v, do, causal=causal)
            for name, a, r in zip(("dq", "dk", "dv"), got, ref):
                if not _close(a, r, rtol=1e-9, atol=1e-11):
                    fails.append(f"gqa {name} vs library autograd shape={(b, h_q, h_kv)} "
                                 f"causal={causal}")
    q = rng.standard_normal((1, 3, 4, 8))
    k = rng.standard_normal((1, 3, 6, 8))
    v = rng.standard_normal((1, 3, 6, 8))
    do = rng.standard_normal((1, 3, 4, 8))
    g1 = impl.gqa_attention_backward(q, k, v, do)
    g2 = impl.attention_backward(q, k, v, do)
    if not all(_close(a, b) for a, b in zip(g1, g2)):
        fails.append("gqa backward with one query head per key/value head")
    return fails


def _scatter_into_pages(k, v, lens, page_size, rng, spare=3):
    """Lay contiguous per-sequence caches k, v [B, h_kv, T, d] out in a pool
    of pages in random order; returns (k_pages, v_pages, block_table). Rows
    past a sequence's length are left as garbage (must not be read)."""
    B, h_kv, T, d = k.shape
    max_pages = -(-T // page_size)
    num_pages = B * max_pages + spare
    perm = rng.permutation(num_pages)
    kp = rng.standard_normal((num_pages, h_kv, page_size, d)) * 50.0   # garbage
    vp = rng.standard_normal((num_pages, h_kv, page_size, d)) * 50.0
    table = np.full((B, max_pages), -1, dtype=np.int64)
    n = 0
    for b in range(B):
        for j in range(-(-int(lens[b]) // page_size)):
            pg = int(perm[n])
            n += 1
            table[b, j] = pg
            rows = slice(j * page_size, min((j + 1) * page_size, int(lens[b])))
            cnt = rows.stop - rows.start
            kp[pg, :, :cnt] = k[b, :, rows]
            vp[pg, :, :cnt] = v[b, :, rows]
    table[table < 0] = int(perm[-1])   # unused entries point at a valid page
    return kp, vp, table


def check_paged(impl):
    import torch
    import torch.nn.functional as F
    fails = []
    rng = _rng(13)
    for (B, h_q, h_kv, T, d, page_size) in ((3, 4, 2, 37, 8, 8), (2, 3, 3, 64, 16, 16), (4, 8, 1, 20, 4, 4)):
        k = rng.standard_normal((B, h_kv, T, d))
        v = rng.standard_normal((B, h_kv, T, d))
        q = rng.standard_normal((B, h_q, d))
        lens = rng.integers(1, T + 1, size=B)
        lens[0] = T
        kp, vp, table = _scatter_into_pages(k, v, lens, page_size, rng)
        o, lse = impl.paged_decode_attention(q, kp, vp, table, lens)
        g = h_q // h_kv
        for b in range(B):
            n = int(lens[b])
            o_ref, l_ref = impl.gqa_attention(q[b:b + 1, :, None, :], k[b:b + 1, :, :n], v[b:b + 1, :, :n])
            if not (_close(o[b], o_ref[0, :, 0]) and _close(lse[b], l_ref[0, :, 0])):
                fails.append(f"paged vs contiguous b={b} shape={(B, h_q, h_kv, T, d, page_size)}")
            kk = torch.from_numpy(np.repeat(k[b:b + 1, :, :n], g, axis=1))
            vv = torch.from_numpy(np.repeat(v[b:b + 1, :, :n], g, axis=1))
            o_lib = F.scaled_dot_product_attention(torch.from_numpy(q[b:b + 1, :, None, :]), kk, vv)
            if not _close(o[b], o_lib.numpy()[0, :, 0], rtol=1e-10, atol=1e-12):
                fails.append(f"paged vs library b={b}")
        # renumbering the pages (and the table with them) changes nothing
        perm = rng.permutation(kp.shape[0])
        inv = np.argsort(perm)
        o2, lse2 = impl.paged_decode_attention(q, kp[perm], vp[perm], inv[table], lens)
        if not (_close(o2, o) and _close(lse2, lse)):
            fails.append("page renumbering must not change the result")
    # a zero length: output 0, lse -inf, other rows unaffected
    k = rng.standard_normal((2, 1, 9, 4))
    v = rng.standard_normal((2, 1, 9, 4))
    q = rng.standard_normal((2, 2, 4))
    kp, vp, table = _scatter_into_pages(k, v, np.array([9, 9]), 4, rng)
    o, lse = impl.paged_decode_attention(q, kp, vp, table, np.array([0, 9]))
    o_full, lse_full = impl.paged_decode_attention(q, kp, vp, table, np.array([9, 9]))
    if not (np.all(o[0] == 0) and np.all(np.isneginf(lse[0])) and _close(o[1], o_full[1])
            and _close(lse[1], lse_full[1])):
        fails.append("zero-length sequence convention")
    return fails


ALL_CHECKS = [
    check_worked_example,
    check_blockwise_equals_full,
    check_bruteforce,
    check_library,
    check_closed_forms,
    check_invariants,
    check_split_merge,
    check_gqa,
    check_backward_library,
    check_backward_finite_difference,
    check_backward_closed_forms,
    check_backward_invariants,
    check_backward_gqa,
    check_paged,
]


def run_all(impl):
    fails = []
    for check in ALL_CHECKS:
        try:
            fails += [f"{check.__name__}: {m}" for m in check(impl)]
        except Exception as exc:  # a mutant may also crash a check
            fails.append(f"{check.__name__}: raised {type(exc).__name__}: {exc}")
    return fails
