"""Blockwise attention with an online softmax, on the CPU in float64 (pin for the oracle).

This is the method the LWM pages run ("Blockwise RingAttention": the sequence is cut
into query and key/value blocks and processed block by block; deep-dive page, section
"RingAttention 为什么必要"), with the running-max / running-sum normaliser of the
blockwise-transformer prior art the pages cite by title ("Blockwise Parallel
Transformer for Large Context Models", "Ring Attention with Blockwise Transformers").
Since the method is exact, its result must not depend on the block sizes or on the
order in which key blocks are visited; tests compare it with the whole-row oracle.
"""

import numpy as np


def forward(q, k, v, seg, block_q, block_k, order="ascending"):
    """One batch row: q, k, v [S, H, D], seg [S]. Returns (out [S,H,D], lse [H,S]).

    ``order``: "ascending" visits key blocks 0, 1, ...; "descending" visits them from
    the diagonal block back to block 0 (the order a ring hands blocks to a device
    holding a later query block).
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    seg = np.asarray(seg)
    S, H, D = q.shape
    scale = 1.0 / np.sqrt(D)
    out = np.zeros((S, H, D))
    lse = np.full((H, S), -np.inf)
    for h in range(H):
        for q0 in range(0, S, block_q):
            q1 = min(S, q0 + block_q)
            rows = np.arange(q0, q1)
            m = np.full(q1 - q0, -np.inf)
            l = np.zeros(q1 - q0)
            acc = np.zeros((q1 - q0, D))
            blocks = list(range(0, q1, block_k))
            if order == "descending":
                blocks = blocks[::-1]
            for k0 in blocks:
                k1 = min(S, k0 + block_k)
                cols = np.arange(k0, k1)
                vis = (seg[cols][None, :] == seg[rows][:, None]) & (seg[rows][:, None] >= 0) \
                    & (cols[None, :] <= rows[:, None])
                s = np.where(vis, (q[rows, h] @ k[k0:k1, h].T) * scale, -np.inf)
                m_new = np.maximum(m, s.max(axis=1))
                live = np.isfinite(m_new)
                both = live & np.isfinite(m)
                with np.errstate(invalid="ignore"):
                    diff = np.where(both, m - m_new, 0.0)
                alpha = np.where(both, np.exp(diff), 0.0)
                p = np.where(vis & live[:, None], np.exp(s - np.where(live, m_new, 0.0)[:, None]), 0.0)
                l = alpha * l + p.sum(axis=1)
                acc = alpha[:, None] * acc + p @ v[k0:k1, h]
                m = np.where(live, m_new, m)
            ok = l > 0
            out[rows[ok], h] = acc[ok] / l[ok][:, None]
            lse[h, rows[ok]] = m[ok] + np.log(l[ok])
    return out, lse
