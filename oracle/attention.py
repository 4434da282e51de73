"""Plain float64 oracle: exact causal, segment-masked softmax attention and its gradients.

Test infrastructure only: the product path never imports this module.

What is computed (LWM, "World Model on Million-Length Video And Language With
Blockwise RingAttention"; charles2530.github.io deep-dive page):
  * exact full softmax attention over the whole sequence, no window and no sparse
    approximation (section "RingAttention 为什么必要");
  * causal, because the model predicts the next token (section "模型结构");
  * masked sequence packing: a packed row holds several documents and the mask lets
    each one attend only to itself (section "Masked sequence packing").

For batch row b, head h and query row i with seg[b,i] >= 0:

    V(i)   = { j : seg[b,j] == seg[b,i] and j <= i }                 (visible keys)
    s_ij   = (q_i . k_j) / sqrt(D)
    lse_i  = log sum_{j in V(i)} exp(s_ij)                           (natural log)
    p_ij   = exp(s_ij - lse_i) for j in V(i), 0 otherwise
    o_i    = sum_j p_ij v_j

and, for an upstream gradient dO of L = sum(dO * O):

    dv_j   = sum_i p_ij do_i
    dp_ij  = do_i . v_j
    delta_i= sum_j p_ij dp_ij
    ds_ij  = p_ij (dp_ij - delta_i)
    dq_i   = (1/sqrt(D)) sum_j ds_ij k_j
    dk_j   = (1/sqrt(D)) sum_i ds_ij q_i

Rows with seg < 0 (padding) see nothing: o = 0, lse = -inf, and they add nothing to
any gradient. The softmax scale is fixed at 1/sqrt(D).

Only the rows are processed in chunks, to bound memory: each query row is still the
plain, whole-row softmax of its definition, and only keys j <= max(row) of a chunk
are formed because every other key is outside every V(i) of the chunk. No online
softmax, blocking over keys or reordering is used here.

Layouts: q, k, v, dout are [B, S, H, D]; seg is [B, S]; lse is returned as [B, H, S].
Inputs are converted to float64 (callers pass the bf16-rounded values so that both
sides see the same numbers).
"""

from __future__ import annotations

import numpy as np

ROW_CHUNK = 1024


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def visible_mask(seg_row, rows):
    """Boolean [len(rows), S] mask: key j is visible from query i.

    j is visible iff seg[j] == seg[i], seg[i] >= 0 and j <= i (same document and
    causal; LWM deep-dive page, sections "Masked sequence packing" and "模型结构").
    """
    seg_row = np.asarray(seg_row)
    rows = np.asarray(rows, dtype=np.int64)
    j = np.arange(seg_row.shape[0])
    si = seg_row[rows][:, None]
    return (seg_row[None, :] == si) & (si >= 0) & (j[None, :] <= rows[:, None])


def _rows_softmax(q_bh, k_bh, seg_row, rows, scale):
    """Scores, probabilities and lse for query rows ``rows`` of one (b, h).

    Returns (p [R, J], lse [R], J) where J = max(rows) + 1 keys are formed.
    """
    J = int(rows.max()) + 1
    mask = visible_mask(seg_row[:J], rows) if J > 0 else np.zeros((len(rows), 0), bool)
    s = (q_bh[rows] @ k_bh[:J].T) * scale
    s = np.where(mask, s, -np.inf)
    has = mask.any(axis=1)
    m = np.where(has, np.max(s, axis=1, initial=-np.inf), 0.0)
    with np.errstate(invalid="ignore"):
        e = np.where(mask, np.exp(s - m[:, None]), 0.0)
    l = e.sum(axis=1)
    lse = np.full(len(rows), -np.inf)
    lse[has] = m[has] + np.log(l[has])
    p = np.zeros_like(s)
    p[has] = e[has] / l[has][:, None]
    return p, lse, J


def _chunks(rows, size=ROW_CHUNK):
    for c in range(0, len(rows), size):
        yield rows[c:c + size]


def attention_forward(q, k, v, seg=None):
    """Full forward pass: returns (out [B,S,H,D], lse [B,H,S]) in float64."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, S, H, D = q.shape
    if seg is None:
        seg = np.zeros((B, S), np.int64)
    seg = np.asarray(seg)
    scale = 1.0 / np.sqrt(D)
    out = np.zeros((B, S, H, D))
    lse = np.full((B, H, S), -np.inf)
    rows_all = np.arange(S)
    for b in range(B):
        for h in range(H):
            for rows in _chunks(rows_all):
                p, l, J = _rows_softmax(q[b, :, h], k[b, :, h], seg[b], rows, scale)
                out[b, rows, h] = p @ v[b, :J, h]
                lse[b, h, rows] = l
    return out, lse


def attention_backward(q, k, v, dout, seg=None):
    """Full gradients (dq, dk, dv), each [B,S,H,D] float64, for L = sum(dout * out)."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, S, H, D = q.shape
    if seg is None:
        seg = np.zeros((B, S), np.int64)
    seg = np.asarray(seg)
    scale = 1.0 / np.sqrt(D)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    rows_all = np.arange(S)
    for b in range(B):
        for h in range(H):
            for rows in _chunks(rows_all):
                p, _, J = _rows_softmax(q[b, :, h], k[b, :, h], seg[b], rows, scale)
                do = dout[b, rows, h]
                dp = do @ v[b, :J, h].T
                delta = np.sum(p * dp, axis=1)
                ds = p * (dp - delta[:, None])
                dq[b, rows, h] = scale * (ds @ k[b, :J, h])
                dk[b, :J, h] += scale * (ds.T @ q[b, rows, h])
                dv[b, :J, h] += p.T @ do
    return dq, dk, dv


def attention_forward_rows(q, k, v, seg, b, rows, heads=None):
    """Forward pass for selected query rows of batch row ``b``.

    Returns (out [R, Hs, D], lse [Hs, R]) for heads ``heads`` (default: all).
    Each row is the same whole-row softmax as in :func:`attention_forward`.
    """
    B, S, H, D = np.shape(q)
    heads = list(range(H)) if heads is None else list(heads)
    rows = np.asarray(rows, dtype=np.int64)
    seg_row = np.zeros(S, np.int64) if seg is None else np.asarray(seg)[b]
    scale = 1.0 / np.sqrt(D)
    out = np.zeros((len(rows), len(heads), D))
    lse = np.zeros((len(heads), len(rows)))
    for hi, h in enumerate(heads):
        qh, kh, vh = _f64(q[b, :, h]), None, None
        J = int(rows.max()) + 1
        kh = _f64(k[b, :J, h])
        vh = _f64(v[b, :J, h])
        for idx in _chunks(np.arange(len(rows)), 256):
            p, l, Jc = _rows_softmax(qh, kh, seg_row, rows[idx], scale)
            out[idx, hi] = p @ vh[:Jc]
            lse[hi, idx] = l
    return out, lse


def attention_backward_rows(q, k, v, dout, seg, b, rows, heads=None):
    """dq for selected query rows of batch row ``b``: [R, Hs, D] float64.

    dq_i needs only row i's own probabilities, so it is exact from the row alone.
    """
    B, S, H, D = np.shape(q)
    heads = list(range(H)) if heads is None else list(heads)
    rows = np.asarray(rows, dtype=np.int64)
    seg_row = np.zeros(S, np.int64) if seg is None else np.asarray(seg)[b]
    scale = 1.0 / np.sqrt(D)
    dq = np.zeros((len(rows), len(heads), D))
    J = int(rows.max()) + 1
    for hi, h in enumerate(heads):
        qh = _f64(q[b, :, h])
        kh = _f64(k[b, :J, h])
        vh = _f64(v[b, :J, h])
        for idx in _chunks(np.arange(len(rows)), 256):
            r = rows[idx]
            p, _, Jc = _rows_softmax(qh, kh, seg_row, r, scale)
            do = _f64(dout[b, r, h])
            dp = do @ vh[:Jc].T
            delta = np.sum(p * dp, axis=1)
            ds = p * (dp - delta[:, None])
            dq[idx, hi] = scale * (ds @ kh[:Jc])
    return dq


def attention_key_grads(q, k, v, dout, seg, b, h, keys):
    """(dk [K, D], dv [K, D]) for selected keys of batch row ``b``, head ``h``.

    dk_j and dv_j sum over every query that sees key j, and each term needs that
    query's whole-row softmax, so every row i >= min(keys) is formed in full.
    """
    B, S, H, D = np.shape(q)
    keys = np.asarray(keys, dtype=np.int64)
    seg_row = np.zeros(S, np.int64) if seg is None else np.asarray(seg)[b]
    scale = 1.0 / np.sqrt(D)
    qh = _f64(q[b, :, h])
    kh = _f64(k[b, :, h])
    vh = _f64(v[b, :, h])
    doh = _f64(dout[b, :, h])
    dk = np.zeros((len(keys), D))
    dv = np.zeros((len(keys), D))
    start = int(keys.min())
    for rows in _chunks(np.arange(start, S)):
        p, _, J = _rows_softmax(qh, kh, seg_row, rows, scale)
        do = doh[rows]
        dp = do @ vh[:J].T
        delta = np.sum(p * dp, axis=1)
        sel = keys < J
        if not sel.any():
            continue
        kk = keys[sel]
        ps = p[:, kk]
        ds = ps * (dp[:, kk] - delta[:, None])
        dk[sel] += scale * (ds.T @ qh[rows])
        dv[sel] += ps.T @ do
    return dk, dv


def credited_pairs(seg):
    """Number of visible (i, j) pairs per head, summed over all batch rows.

    Counts, for every query i with seg >= 0, the keys j <= i of the same segment
    (the definition of V(i) above), using a running count per segment id.
    """
    seg = np.asarray(seg)
    total = 0
    for b in range(seg.shape[0]):
        counts = {}
        for s in seg[b].tolist():
            if s < 0:
                continue
            c = counts.get(s, 0) + 1
            counts[s] = c
            total += c
    return total
