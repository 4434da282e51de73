"""Re-weighted packed cross-entropy (lwm_packed_loss) against the float64 oracle
(oracle/loss_weighting.py), plus the defining property on the GPU itself: a packed
batch gives the loss and gradients of the same documents run non-packed, one per
padded row.

Bars: the loss to 1e-5 relative (the kernel's log-sum-exp is fp32, its sums fp64);
the gradient, stored in bf16, per element within 2^-8 |g| + 1e-6 max|g| of the
oracle (bf16 rounding plus the fp32 softmax).
"""

import numpy as np
import pytest
import torch

import blockwise_ringattention_causal_b300 as lwm
from blockwise_ringattention_causal_b300 import inputs as I
import oracle
from tests._parity import f64

pytestmark = pytest.mark.gpu


def _inputs(lengths, S, V, device, seed, scale=4.0, weights="mask"):
    B = len(lengths)
    w = I.custom(B, S, 1, 128, lengths, seed=seed)
    seg, _ = I.segments(w)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    logits = (torch.randn((B, S, V), generator=g, device=device) * scale).to(torch.bfloat16)
    targets = torch.randint(0, V, (B, S), generator=g, device=device, dtype=torch.int32)
    if weights == "mask":              # no loss on the last token of each document
        wt = np.ones((B, S), np.float32)
        for b, lens in enumerate(lengths):
            ends = np.cumsum(lens) - 1
            wt[b, ends] = 0.0
    else:
        rng = np.random.default_rng(seed)
        wt = (rng.random((B, S)) < 0.8).astype(np.float32) * rng.uniform(0.25, 2.0, (B, S)).astype(np.float32)
    return logits, targets, torch.from_numpy(wt).to(device), torch.from_numpy(seg).to(device)


def _check(logits, targets, wt, seg, what):
    loss, grad, ws = lwm.packed_loss(logits, targets, wt, seg)
    assert lwm.lwm_attn_check(ws) == 0
    ref_loss, ref_grad = oracle.packed_loss(f64(logits), targets.cpu().numpy(), seg.cpu().numpy(),
                                            None if wt is None else wt.cpu().numpy())
    assert abs(float(loss) - ref_loss) <= 1e-5 * abs(ref_loss), f"{what}: {float(loss)} vs {ref_loss}"
    g = f64(grad)
    bound = 2.0 ** -8 * np.abs(ref_grad) + 1e-6 * np.abs(ref_grad).max()
    assert np.all(np.abs(g - ref_grad) <= bound), f"{what}: grad off by {np.max(np.abs(g - ref_grad) - bound):.3e}"
    return float(loss)


@pytest.mark.parametrize("weights", ["mask", "float"])
def test_packed_rows_with_padding(cuda_device, weights):
    lengths = [[300, 1, 250, 100], [700], [5, 3, 400, 7]]     # row 2 ends in padding
    logits, targets, wt, seg = _inputs(lengths, 700, 1000, cuda_device, seed=1, weights=weights)
    _check(logits, targets, wt, seg, f"packed {weights}")


def test_defaults_one_document_per_row(cuda_device):
    logits, targets, _, _ = _inputs([[257], [257]], 257, 264, cuda_device, seed=2)
    loss, grad, ws = lwm.packed_loss(logits, targets)
    assert lwm.lwm_attn_check(ws) == 0
    ref_loss, ref_grad = oracle.packed_loss(f64(logits), targets.cpu().numpy())
    assert abs(float(loss) - ref_loss) <= 1e-5 * abs(ref_loss)
    loss2, none, _ = lwm.packed_loss(logits, targets, grad=False)
    assert none is None and float(loss2) == float(loss)


def test_packed_equals_nonpacked_with_padding_on_the_gpu(cuda_device):
    """The pages' property, on the kernel: pack three documents into one row, or give
    each its own row padded to the longest; same loss, same gradients."""
    lens = [300, 45, 211]
    S = sum(lens)
    V = 512
    logits, targets, wt, seg = _inputs([lens], S, V, cuda_device, seed=3)
    loss_p, grad_p, _ = lwm.packed_loss(logits, targets, wt, seg)
    L = max(lens)
    B = len(lens)
    lg = torch.zeros((B, L, V), dtype=torch.bfloat16, device=cuda_device)
    tg = torch.zeros((B, L), dtype=torch.int32, device=cuda_device)
    wg = torch.zeros((B, L), dtype=torch.float32, device=cuda_device)
    sg = torch.full((B, L), -1, dtype=torch.int32, device=cuda_device)
    o = 0
    for b, n in enumerate(lens):
        lg[b, :n], tg[b, :n], wg[b, :n], sg[b, :n] = logits[0, o:o + n], targets[0, o:o + n], wt[0, o:o + n], 0
        o += n
    loss_u, grad_u, _ = lwm.packed_loss(lg, tg, wg, sg)
    assert abs(float(loss_p) - float(loss_u)) <= 1e-6 * abs(float(loss_u))
    o = 0
    for b, n in enumerate(lens):
        assert torch.equal(grad_p[0, o:o + n], grad_u[b, :n])
        assert torch.all(grad_u[b, n:] == 0)
        o += n


def test_mixed_packing_s64k_rows(cuda_device):
    """The mixed text / image packing of two 64K-token rows (44 documents), V = 4096:
    the whole loss exactly, the gradient on 512 sampled rows of each batch row."""
    w = I.workload(3)
    V = 4096
    logits, targets, wt, seg = _inputs(w.lengths, w.S, V, cuda_device, seed=4)
    loss, grad, ws = lwm.packed_loss(logits, targets, wt, seg)
    assert lwm.lwm_attn_check(ws) == 0
    segn, wn, yn = seg.cpu().numpy(), wt.cpu().numpy(), targets.cpu().numpy()
    # the oracle's loss over every token, in row chunks (float64)
    docs = [(b, s0, s1) for b in range(w.B) for s0, s1 in oracle.documents(segn[b]) if wn[b, s0:s1].sum() > 0]
    total = 0.0
    for b, s0, s1 in docs:
        ce = np.concatenate([oracle.token_cross_entropy(f64(logits[b, c:min(c + 4096, s1)]), yn[b, c:min(c + 4096, s1)])
                             for c in range(s0, s1, 4096)])
        total += float(np.sum(wn[b, s0:s1] * ce)) / float(wn[b, s0:s1].sum()) / len(docs)
    assert abs(float(loss) - total) <= 1e-5 * abs(total)
    rows = I.sample_rows(w.S)
    for b in range(w.B):
        for r in rows:
            d = next((s0, s1) for bb, s0, s1 in docs if bb == b and s0 <= r < s1) if wn[b, r] > 0 else None
            z = f64(logits[b, r])
            if d is None:
                assert torch.all(grad[b, r] == 0)
                continue
            p = np.exp(z - z.max()); p /= p.sum(); p[yn[b, r]] -= 1.0
            ref = wn[b, r] / (float(wn[b, d[0]:d[1]].sum()) * len(docs)) * p
            g = f64(grad[b, r])
            assert np.all(np.abs(g - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6 * np.abs(ref).max()), (b, r)


def test_errors_are_reported(cuda_device):
    logits, targets, wt, seg = _inputs([[100, 100]], 200, 64, cuda_device, seed=5)
    bad = targets.clone()
    bad[0, 10] = 64
    _, _, ws = lwm.packed_loss(logits, bad, wt, seg)
    assert lwm.lwm_attn_check(ws) == 9
    wt2 = wt.clone()
    wt2[0, 10] = 0.0                                   # a target outside [0, V) on an unweighted token is fine
    _, _, ws = lwm.packed_loss(logits, bad, wt2, seg)
    assert lwm.lwm_attn_check(ws) == 0
    bad_seg = seg.clone()
    bad_seg[0, 150:] = 0                               # ids go back down
    _, _, ws = lwm.packed_loss(logits, targets, wt, bad_seg)
    assert lwm.lwm_attn_check(ws) == 4
