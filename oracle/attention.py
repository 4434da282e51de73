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
plain, whole-row softmax of its definition. Of the keys, a chunk forms only the
window [j0, max(row)] outside which the mask shows no visible key for any of its rows
(p = 0 there, exactly). No online softmax, blocking over keys or reordering is used
here.

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

    ``q_bh`` and ``k_bh`` are [S, D] (any float type; the rows used are taken to float64).

    Returns (p [R, J - j0], lse [R], j0, J): J = max(rows) + 1, and [j0, J) holds every
    key that the mask makes visible from at least one of the rows (the first such key
    is j0; keys outside that window are invisible from every row, so their p is 0 and
    they are not formed). p[:, c] belongs to key j0 + c.
    """
    J = int(rows.max()) + 1
    mask = visible_mask(seg_row[:J], rows) if J > 0 else np.zeros((len(rows), 0), bool)
    cols = mask.any(axis=0)
    j0 = int(np.argmax(cols)) if cols.any() else J
    mask = mask[:, j0:]
    s = (_f64(q_bh[rows]) @ _f64(k_bh[j0:J]).T) * scale
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
    return p, lse, j0, J


def _chunk_rows(n_keys):
    """Rows per chunk: at most ROW_CHUNK, and few enough that a chunk's score matrix over
    ``n_keys`` keys holds at most 2^24 entries (memory only; every row is independent)."""
    return max(16, min(ROW_CHUNK, (1 << 24) // max(int(n_keys), 1)))


def _chunks(rows, size=ROW_CHUNK):
    for c in range(0, len(rows), size):
        yield rows[c:c + size]


def _seg_or_zeros(seg, B, S):
    return np.zeros((B, S), np.int64) if seg is None else np.asarray(seg)


def forward_row_block(q, k, v, seg, b, h, rows):
    """out [R, D] and lse [R] of query rows ``rows`` of (b, h): the whole-row softmax of
    each row (the body of :func:`attention_forward`)."""
    B, S, H, D = np.shape(q)
    seg_row = _seg_or_zeros(seg, B, S)[b]
    rows = np.asarray(rows, dtype=np.int64)
    p, lse, j0, J = _rows_softmax(q[b, :, h], k[b, :, h], seg_row, rows, 1.0 / np.sqrt(D))
    return p @ _f64(v[b, j0:J, h]), lse


def backward_row_block(q, k, v, dout, seg, b, h, rows):
    """Gradient terms of query rows ``rows`` of (b, h) (the body of :func:`attention_backward`).

    Returns (dq [R, D], j0, dk_part [J - j0, D], dv_part [J - j0, D]): dq of those rows,
    and their terms of dk_j and dv_j for keys j0 <= j < J (no other key gets any from
    these rows). dk and dv are the sums of these terms over all row blocks.
    """
    B, S, H, D = np.shape(q)
    seg_row = _seg_or_zeros(seg, B, S)[b]
    rows = np.asarray(rows, dtype=np.int64)
    scale = 1.0 / np.sqrt(D)
    p, _, j0, J = _rows_softmax(q[b, :, h], k[b, :, h], seg_row, rows, scale)
    kw, vw = _f64(k[b, j0:J, h]), _f64(v[b, j0:J, h])
    do = _f64(dout[b, rows, h])
    dp = do @ vw.T
    delta = np.sum(p * dp, axis=1)
    ds = p * (dp - delta[:, None])
    return scale * (ds @ kw), j0, scale * (ds.T @ _f64(q[b, rows, h])), p.T @ do


def attention_forward(q, k, v, seg=None):
    """Full forward pass: returns (out [B,S,H,D], lse [B,H,S]) in float64."""
    B, S, H, D = np.shape(q)
    out = np.zeros((B, S, H, D))
    lse = np.full((B, H, S), -np.inf)
    for b in range(B):
        for h in range(H):
            for rows in _chunks(np.arange(S), _chunk_rows(S)):
                out[b, rows, h], lse[b, h, rows] = forward_row_block(q, k, v, seg, b, h, rows)
    return out, lse


def attention_backward(q, k, v, dout, seg=None):
    """Full gradients (dq, dk, dv), each [B,S,H,D] float64, for L = sum(dout * out)."""
    B, S, H, D = np.shape(q)
    dq = np.zeros((B, S, H, D))
    dk = np.zeros((B, S, H, D))
    dv = np.zeros((B, S, H, D))
    for b in range(B):
        for h in range(H):
            for rows in _chunks(np.arange(S), _chunk_rows(S)):
                g, j0, gk, gv = backward_row_block(q, k, v, dout, seg, b, h, rows)
                J = j0 + gk.shape[0]
                dq[b, rows, h] = g
                dk[b, j0:J, h] += gk
                dv[b, j0:J, h] += gv
    return dq, dk, dv


def attention_forward_rows(q, k, v, seg, b, rows, heads=None):
    """Forward pass for selected query rows of batch row ``b``.

    Returns (out [R, Hs, D], lse [Hs, R]) for heads ``heads`` (default: all).
    Each row is the same whole-row softmax as in :func:`attention_forward`.
    """
    B, S, H, D = np.shape(q)
    heads = list(range(H)) if heads is None else list(heads)
    rows = np.asarray(rows, dtype=np.int64)
    out = np.zeros((len(rows), len(heads), D))
    lse = np.zeros((len(heads), len(rows)))
    for hi, h in enumerate(heads):
        for idx in _chunks(np.arange(len(rows)), 256):
            out[idx, hi], lse[hi, idx] = forward_row_block(q, k, v, seg, b, h, rows[idx])
    return out, lse


def attention_backward_rows(q, k, v, dout, seg, b, rows, heads=None):
    """dq for selected query rows of batch row ``b``: [R, Hs, D] float64.

    dq_i needs only row i's own probabilities, so it is exact from the row alone.
    """
    B, S, H, D = np.shape(q)
    heads = list(range(H)) if heads is None else list(heads)
    rows = np.asarray(rows, dtype=np.int64)
    dq = np.zeros((len(rows), len(heads), D))
    for hi, h in enumerate(heads):
        for idx in _chunks(np.arange(len(rows)), 256):
            dq[idx, hi] = backward_row_block(q, k, v, dout, seg, b, h, rows[idx])[0]
    return dq


def attention_key_grads(q, k, v, dout, seg, b, h, keys, row_range=None):
    """(dk [K, D], dv [K, D]) for selected keys of batch row ``b``, head ``h``.

    dk_j and dv_j sum over every query that sees key j, and each term needs that
    query's whole-row softmax (and its delta), so every row i >= min(keys) is formed
    in full; only the selected keys' columns of ds and p enter the sums.
    ``row_range`` = (r0, r1) restricts the sum to queries r0 <= i < r1 (a part of the
    sum; the parts over disjoint ranges add up to the whole).
    """
    B, S, H, D = np.shape(q)
    keys = np.asarray(keys, dtype=np.int64)
    seg_row = _seg_or_zeros(seg, B, S)[b]
    scale = 1.0 / np.sqrt(D)
    start, stop = (int(keys.min()), S) if row_range is None else (max(int(keys.min()), row_range[0]), row_range[1])
    dk = np.zeros((len(keys), D))
    dv = np.zeros((len(keys), D))
    if stop <= start:
        return dk, dv
    for rows in _chunks(np.arange(start, stop), _chunk_rows(stop)):
        p, _, j0, J = _rows_softmax(q[b, :, h], k[b, :, h], seg_row, rows, scale)
        sel = (keys >= j0) & (keys < J)
        if not sel.any():
            continue
        do = _f64(dout[b, rows, h])
        dp = do @ _f64(v[b, j0:J, h]).T
        delta = np.sum(p * dp, axis=1)
        cols = keys[sel] - j0
        ps = p[:, cols]
        ds = ps * (dp[:, cols] - delta[:, None])
        dk[sel] += scale * (ds.T @ _f64(q[b, rows, h]))
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
