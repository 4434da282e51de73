"""Pure-Python attention by explicit loops, for tiny inputs (pin for the oracle).

Written straight from the definition of exact causal attention with a packing mask
(LWM deep-dive page, sections "RingAttention 为什么必要", "模型结构" and "Masked
sequence packing"): query i of document seg[i] attends to keys j <= i of the same
document, with softmax weights exp(q_i.k_j / sqrt(D)). No NumPy, no vectorisation.
"""

import math


def forward(q, k, v, seg):
    """q, k, v: nested lists [S][H][D]; seg: list [S]. Returns (out [S][H][D], lse [H][S])."""
    S, H, D = len(q), len(q[0]), len(q[0][0])
    scale = 1.0 / math.sqrt(D)
    out = [[[0.0] * D for _ in range(H)] for _ in range(S)]
    lse = [[-math.inf] * S for _ in range(H)]
    for h in range(H):
        for i in range(S):
            if seg[i] < 0:
                continue
            keys = [j for j in range(S) if j <= i and seg[j] == seg[i]]
            scores = []
            for j in keys:
                dot = 0.0
                for d in range(D):
                    dot += q[i][h][d] * k[j][h][d]
                scores.append(dot * scale)
            top = max(scores)
            weights = [math.exp(s - top) for s in scores]
            total = sum(weights)
            lse[h][i] = top + math.log(total)
            for j, w in zip(keys, weights):
                for d in range(D):
                    out[i][h][d] += (w / total) * v[j][h][d]
    return out, lse
