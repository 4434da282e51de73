"""Pins for the packed-loss oracle (oracle/loss_weighting.py), against things other than
itself (CPU only):

  * a worked example derived by hand (tests/golden/packed_loss_worked_example.json);
  * the defining property on the pages: the packed, re-weighted loss equals training
    the same documents non-packed, one per row with padding; the non-packed side is
    built explicitly (padded rows) and evaluated with torch's float64 cross-entropy,
    and its gradient by torch autograd;
  * planted mistake: the naive token mean over the packed batch fails that property.
"""

import json
import math
import os

import numpy as np
import torch

import oracle
from oracle import loss_weighting as PL

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "packed_loss_worked_example.json")


def _ev(e):
    return float(eval(str(e), {"__builtins__": {}}, {"ln2": math.log(2), "ln3": math.log(3), "ln4": math.log(4)}))


def test_worked_example():
    g = json.load(open(GOLDEN))
    z = np.array([[_ev(e) for e in r] for r in g["logits"]])[None]
    y = np.array(g["targets"])[None]
    seg = np.array(g["seg"])[None]
    loss, grad = PL.packed_loss(z, y, seg)
    assert abs(loss - _ev(g["loss"])) < 1e-14
    np.testing.assert_allclose(grad[0], np.array([[_ev(e) for e in r] for r in g["dlogits"]]), atol=1e-15)
    assert abs(loss - _ev(g["naive_token_mean"])) > 1e-3


def _random_packing(rng, B, S):
    seg = np.full((B, S), -1)
    for b in range(B):
        i, d = 0, 0
        real = S - int(rng.integers(0, S // 4))
        while i < real:
            L = min(int(rng.integers(1, S // 3)), real - i)
            seg[b, i:i + L] = d
            i += L
            d += 1
    return seg


def _nonpacked_padded(z, y, seg, w):
    """Every document as its own padded row; row loss = weighted mean over its tokens,
    batch loss = mean over rows with any weight. torch float64 with autograd."""
    docs = [(b, s0, s1) for b in range(seg.shape[0]) for s0, s1 in PL.documents(seg[b])]
    L = max(s1 - s0 for _, s0, s1 in docs)
    V = z.shape[2]
    zt = torch.tensor(z, dtype=torch.float64, requires_grad=True)
    rows = []
    for b, s0, s1 in docs:
        n = s1 - s0
        pad_z = torch.zeros((L - n, V), dtype=torch.float64)
        rz = torch.cat([zt[b, s0:s1], pad_z])
        ry = torch.cat([torch.tensor(y[b, s0:s1]), torch.zeros(L - n, dtype=torch.long)])
        rw = torch.cat([torch.tensor(w[b, s0:s1]), torch.zeros(L - n, dtype=torch.float64)])
        ce = torch.nn.functional.cross_entropy(rz, ry, reduction="none")
        if float(rw.sum()) > 0:
            rows.append((rw * ce).sum() / rw.sum())
    loss = torch.stack(rows).mean()
    loss.backward()
    return float(loss.detach()), zt.grad.numpy()


def test_packed_equals_nonpacked_with_padding():
    rng = np.random.default_rng(0)
    for trial in range(6):
        B, S, V = 2, 40, 7
        seg = _random_packing(rng, B, S)
        z = rng.standard_normal((B, S, V)) * 3
        y = rng.integers(0, V, size=(B, S))
        w = (rng.random((B, S)) < 0.7).astype(np.float64) * rng.uniform(0.5, 2.0, (B, S))
        if trial == 0:
            w[:] = 1.0
        loss, grad = PL.packed_loss(z, y, seg, w)
        ref_loss, ref_grad = _nonpacked_padded(z, y, seg, w)
        assert abs(loss - ref_loss) < 1e-12
        np.testing.assert_allclose(grad, ref_grad, atol=1e-14)
        # planted: the naive token mean over the packed batch is not the same loss
        valid = (seg >= 0)
        ce = PL.token_cross_entropy(z.reshape(-1, V), y.reshape(-1)).reshape(B, S)
        naive = float((w * ce * valid).sum() / (w * valid).sum())
        assert abs(naive - ref_loss) > 1e-4


def test_token_cross_entropy_matches_torch():
    rng = np.random.default_rng(1)
    z = rng.standard_normal((50, 300)) * 10
    y = rng.integers(0, 300, 50)
    ref = torch.nn.functional.cross_entropy(torch.tensor(z), torch.tensor(y), reduction="none").numpy()
    np.testing.assert_allclose(PL.token_cross_entropy(z, y), ref, atol=1e-12)


def test_exported():
    assert oracle.packed_loss is PL.packed_loss
