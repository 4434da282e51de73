"""Plain float64 oracle of the packed-loss re-weighting (test infrastructure only).

What the pages fix (LWM deep-dive page, section "Masked sequence packing"): packing
puts several samples in one row; besides the attention mask, LWM re-weights the loss
so that it equals training the same samples non-packed, one per row with padding
(item 2 of the section's list of what LWM does). The reason given in the same section
(item 2 of its list of problems): in a packed row the token-count of long video
samples would drown the loss of short answers.

Reading (the pages give no formula): in non-packed + padding training each sample is
its own row and the row's loss is the mean of its token losses over its own loss
tokens (padding and unweighted tokens excluded); the batch loss is the mean over the
rows (samples) that have any loss token. A token-mean over the whole packed batch
would weight samples by their token counts, which is what the pages say must be
avoided. With per-token weights w_t >= 0 (0 = no loss on t) and the token loss
l_t = cross-entropy of the logits z_t against target y_t:

    loss = (1 / N) sum_d ( sum_{t in d} w_t l_t / sum_{t in d} w_t ),
    N    = number of documents d with sum_{t in d} w_t > 0,
    l_t  = log sum_v exp(z_t[v]) - z_t[y_t],

and its gradient dloss/dz_t = w_t / (N sum_{t' in d} w_t') (softmax(z_t) - onehot(y_t)).
Documents are the contiguous runs of equal seg >= 0 of a row (as for the attention);
seg < 0 (padding) carries no loss.
"""

from __future__ import annotations

import numpy as np


def token_cross_entropy(logits, targets):
    """l_t = log sum_v exp(z_t[v]) - z_t[y_t] for logits [N, V] and targets [N] (float64)."""
    z = np.asarray(logits, dtype=np.float64)
    y = np.asarray(targets, dtype=np.int64)
    m = z.max(axis=1)
    lse = m + np.log(np.exp(z - m[:, None]).sum(axis=1))
    return lse - z[np.arange(len(y)), y]


def documents(seg_row):
    """[(start, end)) of the contiguous runs of equal seg >= 0 of one row."""
    seg_row = np.asarray(seg_row)
    out, i, S = [], 0, len(seg_row)
    while i < S:
        j = i
        while j < S and seg_row[j] == seg_row[i]:
            j += 1
        if seg_row[i] >= 0:
            out.append((i, j))
        i = j
    return out


def packed_loss(logits, targets, seg=None, weight=None):
    """(loss, dlogits [B, S, V]) of the re-weighted packed loss, float64.

    logits [B, S, V]; targets [B, S]; seg [B, S] (None: one document per row);
    weight [B, S] (None: 1 on every token of a document).
    """
    z = np.asarray(logits, dtype=np.float64)
    B, S, V = z.shape
    y = np.asarray(targets, dtype=np.int64)
    seg = np.zeros((B, S), np.int64) if seg is None else np.asarray(seg)
    w = np.ones((B, S)) if weight is None else np.asarray(weight, dtype=np.float64)
    docs = []
    for b in range(B):
        for s0, s1 in documents(seg[b]):
            if w[b, s0:s1].sum() > 0:
                docs.append((b, s0, s1))
    N = len(docs)
    loss = 0.0
    grad = np.zeros_like(z)
    for b, s0, s1 in docs:
        zt, yt, wt = z[b, s0:s1], y[b, s0:s1], w[b, s0:s1]
        nd = wt.sum()
        loss += float(np.sum(wt * token_cross_entropy(zt, yt))) / nd / N
        p = np.exp(zt - zt.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        p[np.arange(len(yt)), yt] -= 1.0
        grad[b, s0:s1] = (wt / (nd * N))[:, None] * p
    return loss, grad
