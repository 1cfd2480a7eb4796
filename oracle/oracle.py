"""Float64 CPU oracle for exact attention: TEST INFRASTRUCTURE ONLY.

This module is the correctness reference for the GPU kernels. It is plain,
slow and written to be checked by eye against the pages it follows. Only the
test suite, the smoke check and the benchmark's CPU-baseline leg may import
it; the product path (the CUDA library and its binding) never calls it and
shares no code with it.

Pages followed (cited by page title and section):

* "IO-Aware Attention: Tiling the Score Matrix Without Materializing It"
  (mercemay.com) -- section "Softmax over blocks, exactly": the running
  maximum / running sum / rescaled accumulator recurrence for one query row,
  final output o/l; section "Parallelism and the cost of the split": key
  partitions each give a partial (max, sum, output) that are merged with the
  same rescaling; section "What has to stay in fast memory": the per-row
  normalisation constants kept for the backward pass (here: logsumexp).
* "E8.1 IO-aware attention" (coursefy.online) -- "Part 2. Do it in code":
  standard_attention materialises the whole score vector, online_attention
  walks key blocks of size `block` (block < 1 is a ValueError).
* "FlashAttention IO-aware tiling lab" (parsercheat.com) -- the definition
  S = QK^T / sqrt(d), P = softmax(S), O = PV and the kernel phases.
* "Attention and Its Computational Cost" (programmer.ie, Inference ch. 8) --
  section "What is being computed": per head Q is T_q x d, K and V are
  T_kv x d, over B sequences and h heads; causal: position i sees keys up to
  and including itself.
* Paged KV cache: "Attention and Its Computational Cost", section "The other
  shape: one query, many keys" names paging of the cache (with batching,
  grouped-query attention and quantisation) among the ways serving systems
  manage its size, without a layout. The oracle takes the plainest reading:
  a sequence's cache is the concatenation of the pages its block table
  lists, cut at its length; decode attends over exactly those keys
  (paged_decode_attention).
* Backward pass: "IO-Aware Attention: Tiling the Score Matrix Without
  Materializing It", section "What has to stay in fast memory" says only that
  the backward pass recomputes the softmax output from the saved Q, K, V and
  the per-row constants. The gradients themselves are not printed; the
  oracle takes the plainest reading, the derivative of the forward above
  written out by the chain rule (attention_backward).

Readings where the pages are silent:

* Causal alignment when T_q != T_kv: bottom-right. Query row i may see key j
  iff j <= i + (T_kv - T_q). For T_q == T_kv this is the pages' definition
  (row i, counted from 1, sees the first i keys); for one query against a
  cache it sees every key.
* lse is the natural log of sum_j exp(scale * q_i . k_j), in the units of
  the scaled scores (the per-row normaliser the pages keep for the backward).
* The scale is applied to the dot product (scores = k @ q / sqrt(d)); callers
  may pass any finite scale, default 1/sqrt(d).

Parity pins: every function here is pinned by tests in tests/test_oracle.py
against values the pages print, closed forms, invariants, a brute force and a
library routine; none is "parity unpinned".
"""

from __future__ import annotations

import math

import numpy as np

__all__ = [
    "standard_attention",
    "standard_attention_row",
    "online_attention",
    "online_softmax_states",
    "split_partials",
    "merge_partials",
    "split_kv_attention",
    "causal_visible",
    "gqa_attention",
    "attention_backward",
    "gqa_attention_backward",
    "paged_decode_attention",
]


def causal_visible(t_q: int, t_kv: int) -> np.ndarray:
    """Boolean [t_q, t_kv] mask, True where key j is visible to query row i.

    Bottom-right alignment: j <= i + (t_kv - t_q). Follows "Attention and Its
    Computational Cost", section "What is being computed" (position i sees
    the keys up to itself) extended to t_q <= t_kv.
    """
    i = np.arange(t_q)[:, None]
    j = np.arange(t_kv)[None, :]
    return j <= i + (t_kv - t_q)


def _default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)


def standard_attention(q, k, v, scale=None, causal=False, rows=None):
    """Materialising attention, float64: returns (O, lse).

    Shapes: q [..., T_q, d], k [..., T_kv, d], v [..., T_kv, d_v]; leading
    dims (batch, heads) must agree. Per head it forms the whole score matrix
    S = scale * Q K^T, masks it (causal), takes m = rowmax(S),
    P = exp(S - m), l = rowsum(P), O = (P V) / l and lse = m + ln(l).

    `rows`, if given, is a 1-D array of query-row indices; only those rows
    are computed (their causal visibility still uses the absolute index), so
    single rows of a very long sequence can be checked one by one.

    Follows the FlashAttention tiling lab's definition (S = QK^T/sqrt(d),
    P = softmax(S), O = PV), "E8.1 IO-aware attention" Part 2
    (standard_attention materialises the scores) and "Attention and Its
    Computational Cost", section "What is being computed".
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    if q.ndim < 2 or k.ndim != q.ndim or v.ndim != q.ndim:
        raise ValueError("q, k, v must have the same rank >= 2")
    t_q, d = q.shape[-2], q.shape[-1]
    t_kv = k.shape[-2]
    if k.shape[-1] != d or v.shape[-2] != t_kv:
        raise ValueError("shape mismatch between q, k and v")
    if t_kv < 1:
        raise ValueError("softmax over zero keys is undefined")
    if causal and t_q > t_kv:
        raise ValueError("causal attention needs T_q <= T_kv")
    if scale is None:
        scale = _default_scale(d)
    lead = q.shape[:-2]
    if k.shape[:-2] != lead or v.shape[:-2] != lead:
        raise ValueError("leading (batch, head) dims must agree")

    row_idx = np.arange(t_q) if rows is None else np.asarray(rows, dtype=np.int64)
    n_rows = row_idx.shape[0]
    out = np.empty(lead + (n_rows, v.shape[-1]), dtype=np.float64)
    lse = np.empty(lead + (n_rows,), dtype=np.float64)
    if causal:
        visible = (np.arange(t_kv)[None, :]
                   <= row_idx[:, None] + (t_kv - t_q))
    for idx in np.ndindex(*lead):
        qh = q[idx][row_idx]            # [n_rows, d]
        s = scale * (qh @ k[idx].T)     # the materialised score matrix
        if causal:
            s = np.where(visible, s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)               # the materialised probabilities
        l = p.sum(axis=1, keepdims=True)
        out[idx] = (p @ v[idx]) / l
        lse[idx] = (m + np.log(l))[:, 0]
    return out, lse


def standard_attention_row(q, k, v, scale=None):
    """One query row: softmax(K q * scale) @ V with the full score vector.

    The single-query form of "E8.1 IO-aware attention" Part 2
    (standard_attention(q, K, V)). Returns (o [d_v], lse).
    """
    q = np.asarray(q, dtype=np.float64)
    o, lse = standard_attention(q[None, :], k, v, scale=scale)
    return o[0], float(lse[0])


def online_softmax_states(scores, block):
    """Running (m, l) after each block of a score row, float64.

    The state update of "IO-Aware Attention: Tiling the Score Matrix Without
    Materializing It", section "Softmax over blocks, exactly":
    m_i = max(m_{i-1}, max of block i); l_i = e^{m_{i-1}-m_i} l_{i-1} +
    sum over block i of e^{s_j - m_i}. Starts from m = -inf, l = 0.
    """
    if block < 1:
        raise ValueError("block must be at least 1")
    s = np.asarray(scores, dtype=np.float64)
    m, l = -np.inf, 0.0
    states = []
    for start in range(0, s.shape[0], block):
        sb = s[start:start + block]
        m_new = max(m, float(sb.max()))
        l = l * math.exp(m - m_new) + float(np.exp(sb - m_new).sum())
        m = m_new
        states.append((m, l))
    return states


def online_attention(q, k, v, block, scale=None, return_state=False):
    """Block-wise exact attention for one query row, float64.

    Walks the keys in blocks of `block`, keeping only the running maximum m,
    running sum l and running weighted value sum o; when a block raises the
    maximum, the old l and o are multiplied by e^{m_old - m_new} before the
    block's terms are added; the result is o / l. Follows "IO-Aware
    Attention ...", section "Softmax over blocks, exactly" and "E8.1
    IO-aware attention" Part 2 (online_attention; block < 1 -> ValueError).
    With return_state, returns (o/l, m, l, o) so partials can be merged.
    """
    if block < 1:
        raise ValueError("block must be at least 1")
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    if scale is None:
        scale = _default_scale(q.shape[0])
    n = k.shape[0]
    m, l, o = -np.inf, 0.0, np.zeros(v.shape[1], dtype=np.float64)
    for start in range(0, n, block):
        kb = k[start:start + block]
        vb = v[start:start + block]
        s = scale * (kb @ q)                 # this block's scores only
        m_new = max(m, float(s.max()))
        alpha = math.exp(m - m_new)          # <= 1; rescales the old state
        p = np.exp(s - m_new)
        l = l * alpha + float(p.sum())
        o = o * alpha + p @ vb
        m = m_new
    if return_state:
        return o / l, m, l, o
    return o / l


def split_partials(q, k, v, num_splits, scale=None):
    """Per-partition partial state (m_s, l_s, o_s) of one query row.

    Key partition s covers [s*L, min((s+1)*L, n)) with L = ceil(n / S); an
    empty partition gives (m=-inf, l=0, o=0). Each partial is computed over
    its keys with the materialised softmax (the partition is one block).
    Follows "IO-Aware Attention ...", section "Parallelism and the cost of
    the split" (each of P key partitions produces a partial output and a
    partial normaliser).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    if num_splits < 1:
        raise ValueError("num_splits must be at least 1")
    if scale is None:
        scale = _default_scale(q.shape[0])
    n = k.shape[0]
    chunk = -(-n // num_splits)
    ms, ls, os_ = [], [], []
    for s in range(num_splits):
        lo, hi = s * chunk, min((s + 1) * chunk, n)
        if lo >= hi:
            ms.append(-np.inf)
            ls.append(0.0)
            os_.append(np.zeros(v.shape[1]))
            continue
        sc = scale * (k[lo:hi] @ q)
        m = float(sc.max())
        p = np.exp(sc - m)
        ms.append(m)
        ls.append(float(p.sum()))
        os_.append(p @ v[lo:hi])
    return np.array(ms), np.array(ls), np.array(os_)


def merge_partials(ms, ls, os_):
    """Exact merge of partition partials: returns (o, lse).

    M = max_s m_s; weights w_s = e^{m_s - M} (0 for an empty partition);
    L = sum_s w_s l_s; o = sum_s w_s o_s / L; lse = M + ln L. This is the
    rescaling recurrence applied across partitions ("IO-Aware Attention
    ...", section "Parallelism and the cost of the split").
    """
    ms = np.asarray(ms, dtype=np.float64)
    ls = np.asarray(ls, dtype=np.float64)
    os_ = np.asarray(os_, dtype=np.float64)
    big_m = float(ms.max())
    w = np.where(np.isneginf(ms), 0.0, np.exp(ms - big_m))
    big_l = float((w * ls).sum())
    o = (w[:, None] * os_).sum(axis=0) / big_l
    return o, big_m + math.log(big_l)


def split_kv_attention(q, k, v, num_splits, scale=None):
    """Split-KV attention of one query row: partials then exact merge."""
    return merge_partials(*split_partials(q, k, v, num_splits, scale=scale))


def gqa_attention(q, k, v, scale=None, causal=False, rows=None):
    """Grouped-query attention, float64: returns (O, lse).

    q: [B, h_q, T_q, d]; k, v: [B, h_kv, T_kv, d] with h_q a multiple of
    h_kv. Query head i attends with key/value head i // (h_q // h_kv): a group
    of h_q/h_kv query heads shares one cached key/value head ("Attention and
    Its Computational Cost", section "The other shape: one query, many keys":
    grouped-query attention reduces the number of key and value heads and so
    the factor of h in the cache read). Each query head is then plain
    standard_attention against its key/value head.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be [B, h, T, d]")
    h_q, h_kv = q.shape[1], k.shape[1]
    if h_kv < 1 or h_q % h_kv != 0:
        raise ValueError("h_q must be a positive multiple of h_kv")
    group = h_q // h_kv
    outs, lses = [], []
    for i in range(h_q):
        o, l = standard_attention(q[:, i], k[:, i // group], v[:, i // group], scale=scale,
                                  causal=causal, rows=rows)
        outs.append(o)
        lses.append(l)
    return np.stack(outs, axis=1), np.stack(lses, axis=1)


def attention_backward(q, k, v, do, scale=None, causal=False):
    """Gradients of attention, float64: returns (dQ, dK, dV).

    The derivative of O = softmax(scale * Q K^T [masked]) V with respect to
    Q, K and V, given the incoming gradient dO (same shape as O), by the
    chain rule through the materialised forward of standard_attention:

        P   = softmax of the masked scaled scores, row by row
        dV  = P^T dO
        dP  = dO V^T
        dS  = P * (dP - rowsum(P * dP))      (softmax Jacobian, row by row)
        dQ  = scale * dS K
        dK  = scale * dS^T Q

    Masked entries have P = 0 and so dS = 0. The pages state that the
    backward pass recomputes P from Q, K, V and the saved row constants
    ("IO-Aware Attention: Tiling the Score Matrix Without Materializing It",
    section "What has to stay in fast memory") but print no gradient
    formulas; these are the calculus of the forward definition.

    Shapes: q [..., T_q, d], k and v [..., T_kv, d], do [..., T_q, d].
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    if q.ndim < 2 or k.ndim != q.ndim or v.ndim != q.ndim or do.shape[:-1] != q.shape[:-1]:
        raise ValueError("q, k, v, do must have the same rank >= 2 and do the rows of q")
    t_q, d = q.shape[-2], q.shape[-1]
    t_kv = k.shape[-2]
    if k.shape[-1] != d or v.shape[-2] != t_kv or do.shape[-1] != v.shape[-1]:
        raise ValueError("shape mismatch between q, k, v and do")
    if t_kv < 1:
        raise ValueError("softmax over zero keys is undefined")
    if causal and t_q > t_kv:
        raise ValueError("causal attention needs T_q <= T_kv")
    if scale is None:
        scale = _default_scale(d)
    lead = q.shape[:-2]
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    visible = causal_visible(t_q, t_kv) if causal else None
    for idx in np.ndindex(*lead):
        s = scale * (q[idx] @ k[idx].T)
        if causal:
            s = np.where(visible, s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        p = e / e.sum(axis=1, keepdims=True)
        dv[idx] = p.T @ do[idx]
        dp = do[idx] @ v[idx].T
        ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
        dq[idx] = scale * (ds @ k[idx])
        dk[idx] = scale * (ds.T @ q[idx])
    return dq, dk, dv


def gqa_attention_backward(q, k, v, do, scale=None, causal=False):
    """Gradients of grouped-query attention, float64: returns (dQ, dK, dV).

    q, do: [B, h_q, T_q, d]; k, v: [B, h_kv, T_kv, d]. Query head i reads
    key/value head i // (h_q // h_kv) (gqa_attention), so a key/value head's
    gradient is the sum of the gradients its query heads send it; each query
    head's own gradients are attention_backward against that head.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4 or do.shape != q.shape:
        raise ValueError("q, do must be [B, h_q, T_q, d] and k, v [B, h_kv, T_kv, d]")
    h_q, h_kv = q.shape[1], k.shape[1]
    if h_kv < 1 or h_q % h_kv != 0:
        raise ValueError("h_q must be a positive multiple of h_kv")
    group = h_q // h_kv
    dq = np.empty_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for i in range(h_q):
        j = i // group
        dqi, dki, dvi = attention_backward(q[:, i], k[:, j], v[:, j], do[:, i], scale=scale,
                                           causal=causal)
        dq[:, i] = dqi
        dk[:, j] += dki
        dv[:, j] += dvi
    return dq, dk, dv


def paged_decode_attention(q, k_pages, v_pages, block_table, seq_lens, scale=None):
    """Decode (one query row per sequence and head) against a paged cache,
    float64: returns (O [B, h_q, d], lse [B, h_q]).

    q: [B, h_q, d]; k_pages, v_pages: [num_pages, h_kv, page_size, d] (a
    pool of fixed-size pages, each holding page_size consecutive cache rows
    of every key/value head); block_table: [B, max_pages] page indices;
    seq_lens: [B] cache lengths. Sequence b's keys are rows 0..n_b-1 of the
    concatenation of pages block_table[b, 0], block_table[b, 1], ... (for
    the heads), and query head i reads key/value head i // (h_q // h_kv).
    Each row is then plain attention of one query against those keys
    (standard_attention_row). A sequence of length 0 has no keys: its
    output is 0 and its lse is -inf (the softmax over nothing has no value;
    this is the oracle's convention, matched by the kernels).

    The pages name paging among the cache-management techniques of serving
    ("Attention and Its Computational Cost", section "The other shape: one
    query, many keys") without a layout; this gather is the plainest reading.
    """
    q = np.asarray(q, dtype=np.float64)
    kp = np.asarray(k_pages, dtype=np.float64)
    vp = np.asarray(v_pages, dtype=np.float64)
    table = np.asarray(block_table, dtype=np.int64)
    lens = np.asarray(seq_lens, dtype=np.int64)
    if q.ndim != 3 or kp.ndim != 4 or vp.shape != kp.shape:
        raise ValueError("q must be [B, h_q, d] and the page pools [num_pages, h_kv, page_size, d]")
    B, h_q, d = q.shape
    num_pages, h_kv, page_size, dk = kp.shape
    if dk != d or h_kv < 1 or h_q % h_kv != 0:
        raise ValueError("head width or grouping mismatch")
    if table.ndim != 2 or table.shape[0] != B or lens.shape != (B,):
        raise ValueError("block_table must be [B, max_pages] and seq_lens [B]")
    if (lens < 0).any() or (lens > table.shape[1] * page_size).any():
        raise ValueError("a length exceeds the pages its block table can hold")
    group = h_q // h_kv
    out = np.zeros((B, h_q, d), dtype=np.float64)
    lse = np.full((B, h_q), -np.inf, dtype=np.float64)
    for b in range(B):
        n = int(lens[b])
        if n == 0:
            continue
        n_pages = -(-n // page_size)
        pages = table[b, :n_pages]
        if (pages < 0).any() or (pages >= num_pages).any():
            raise ValueError("block table entry outside the page pool")
        for i in range(h_q):
            j = i // group
            keys = np.concatenate([kp[p, j] for p in pages], axis=0)[:n]
            vals = np.concatenate([vp[p, j] for p in pages], axis=0)[:n]
            out[b, i], lse[b, i] = standard_attention_row(q[b, i], keys, vals, scale=scale)
    return out, lse
