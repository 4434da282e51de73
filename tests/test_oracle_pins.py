"""Pins for the float64 oracle, against things other than itself (CPU only).

  * a hand-derived worked example (tests/golden/worked_example_s3_d4.json);
  * brute force with pure-Python loops on tiny inputs;
  * finite differences of L = sum(dO * O) for the analytic gradients;
  * a library routine on special cases: torch's scaled_dot_product_attention in
    float64 with autograd, on causal and on packed (boolean-mask) rows;
  * closed forms (length-1 documents, constant scores -> prefix mean, one dominant key);
  * invariants (packing = documents run alone, block-size and block-order independence
    of the blockwise online softmax, shift invariances, gradient sum rules);
  * planted mistakes: a wrong mask, a wrong scale or a wrong gradient in a copy of the
    oracle must make at least one pin fail.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as OA
from tests import _blockwise_cpu as BW
from tests import _bruteforce as BF

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, rng):
    return rng.standard_normal(shape)


def _random_segments(S, rng, allow_pad=True):
    """Random contiguous documents (ids 0,1,2..) plus optionally a trailing pad run."""
    seg = np.empty(S, np.int64)
    i, d = 0, 0
    pad = int(rng.integers(0, max(1, S // 4))) if allow_pad and rng.random() < 0.5 else 0
    real = S - pad
    while i < real:
        L = int(rng.integers(1, max(2, real // 2 + 1)))
        L = min(L, real - i)
        seg[i:i + L] = d
        i += L
        d += 1
    seg[real:] = -1
    return seg


def _eval(expr):
    if isinstance(expr, (int, float)):
        return float(expr)
    return float(eval(expr, {"__builtins__": {}}, {"ln2": math.log(2), "ln3": math.log(3), "ln6": math.log(6)}))


def _arr(x):
    return np.array([[_eval(e) for e in row] for row in x]) if isinstance(x[0], list) else np.array([_eval(e) for e in x])


# ----------------------------------------------------------------------------- golden

def test_worked_example_golden():
    g = json.load(open(os.path.join(GOLDEN, "worked_example_s3_d4.json")))
    q = _arr(g["q"])[None, :, None, :]
    k = _arr(g["k"])[None, :, None, :]
    v = _arr(g["v"])[None, :, None, :]
    do = _arr(g["dout"])[None, :, None, :]
    for case in g["cases"]:
        seg = np.array(case["seg"])[None]
        out, lse = oracle.attention_forward(q, k, v, seg)
        np.testing.assert_allclose(out[0, :, 0], _arr(case["out"]), atol=1e-13)
        np.testing.assert_allclose(lse[0, 0], _arr(case["lse"]), atol=1e-13)
        dq, dk, dv = oracle.attention_backward(q, k, v, do, seg)
        np.testing.assert_allclose(dq[0, :, 0], _arr(case["dq"]), atol=1e-13)
        np.testing.assert_allclose(dk[0, :, 0], _arr(case["dk"]), atol=1e-13)
        np.testing.assert_allclose(dv[0, :, 0], _arr(case["dv"]), atol=1e-13)


# ----------------------------------------------------------------------------- brute force

@pytest.mark.parametrize("trial", range(12))
def test_brute_force_forward(trial):
    rng = np.random.default_rng(100 + trial)
    S = int(rng.integers(1, 25))
    D = [1, 4, 8][trial % 3]
    H = 1 + trial % 2
    seg = _random_segments(S, rng)
    q, k, v = (_rand((1, S, H, D), rng) for _ in range(3))
    out, lse = oracle.attention_forward(q, k, v, seg[None])
    bo, bl = BF.forward(q[0].tolist(), k[0].tolist(), v[0].tolist(), seg.tolist())
    np.testing.assert_allclose(out[0], np.array(bo), atol=1e-12, rtol=0)
    np.testing.assert_array_equal(np.isinf(lse[0]), np.isinf(np.array(bl)))
    fin = np.isfinite(lse[0])
    np.testing.assert_allclose(lse[0][fin], np.array(bl)[fin], atol=1e-12, rtol=0)


# ----------------------------------------------------------------------------- finite differences

def _loss(q, k, v, do, seg):
    out, _ = oracle.attention_forward(q, k, v, seg)
    return float(np.sum(out * do))


@pytest.mark.parametrize("trial", range(4))
def test_finite_differences(trial):
    rng = np.random.default_rng(200 + trial)
    S, H, D = [5, 9, 16, 12][trial], 1 + trial % 2, [3, 4, 2, 5][trial]
    seg = _random_segments(S, rng)[None]
    q, k, v, do = (_rand((1, S, H, D), rng) for _ in range(4))
    dq, dk, dv = oracle.attention_backward(q, k, v, do, seg)
    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            lp = _loss(args["q"], args["k"], args["v"], do, seg)
            args[name] = xm
            lm = _loss(args["q"], args["k"], args["v"], do, seg)
            num[idx] = (lp - lm) / (2 * h)
        err = np.linalg.norm(num - g) / max(np.linalg.norm(g), 1e-30)
        assert err < 1e-6, (name, err)


# ----------------------------------------------------------------------------- library routine

def _sdpa(q, k, v, seg):
    """torch SDPA in float64 with an explicit boolean mask built from seg (batch row 0)."""
    S = q.shape[1]
    i = torch.arange(S)[:, None]
    j = torch.arange(S)[None, :]
    st = torch.as_tensor(seg[0])
    allowed = (st[None, :] == st[:, None]) & (j <= i)
    qt, kt, vt = (torch.tensor(x[0].transpose(1, 0, 2), requires_grad=True) for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=allowed)
    return qt, kt, vt, out


@pytest.mark.parametrize("packed", [False, True])
def test_torch_sdpa_special_case(packed):
    rng = np.random.default_rng(300 + packed)
    S, H, D = 200, 3, 16
    seg = np.zeros((1, S), np.int64)
    if packed:
        seg[0] = np.repeat(np.arange(4), [37, 80, 1, 82])
    q, k, v, do = (_rand((1, S, H, D), rng) for _ in range(4))
    out, lse = oracle.attention_forward(q, k, v, seg)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, seg)
    qt, kt, vt, ot = _sdpa(q, k, v, seg)
    np.testing.assert_allclose(out[0].transpose(1, 0, 2), ot.detach().numpy(), atol=1e-12)
    ot.backward(torch.tensor(do[0].transpose(1, 0, 2)))
    for mine, ref in ((dq, qt), (dk, kt), (dv, vt)):
        np.testing.assert_allclose(mine[0].transpose(1, 0, 2), ref.grad.numpy(), atol=1e-11)
    # lse against torch.logsumexp over the same masked scores
    st = torch.as_tensor(seg[0])
    i = torch.arange(S)[:, None]
    j = torch.arange(S)[None, :]
    allowed = (st[None, :] == st[:, None]) & (j <= i)
    sc = torch.einsum("hid,hjd->hij", torch.tensor(q[0].transpose(1, 0, 2)),
                      torch.tensor(k[0].transpose(1, 0, 2))) / math.sqrt(D)
    ref_lse = torch.logsumexp(sc.masked_fill(~allowed, -math.inf), dim=-1)
    np.testing.assert_allclose(lse[0], ref_lse.numpy(), atol=1e-12)


# ----------------------------------------------------------------------------- closed forms

def test_length_one_documents_return_own_value():
    rng = np.random.default_rng(7)
    S, H, D = 10, 2, 8
    seg = np.arange(S)[None]                       # every token its own document
    q, k, v = (_rand((1, S, H, D), rng) for _ in range(3))
    out, lse = oracle.attention_forward(q, k, v, seg)
    np.testing.assert_allclose(out, v, atol=1e-14)
    s_ii = np.einsum("bshd,bshd->bhs", q, k) / math.sqrt(D)
    np.testing.assert_allclose(lse, s_ii, atol=1e-14)


def test_constant_scores_give_prefix_mean():
    rng = np.random.default_rng(8)
    S, H, D = 40, 2, 4
    seg = np.repeat([0, 1, 2], [10, 17, 13])[None]
    pos = np.concatenate([np.arange(10), np.arange(17), np.arange(13)])
    q = np.zeros((1, S, H, D))
    k, v = _rand((1, S, H, D), rng), _rand((1, S, H, D), rng)
    out, lse = oracle.attention_forward(q, k, v, seg)
    starts = np.array([0] * 10 + [10] * 17 + [27] * 13)
    for i in range(S):
        np.testing.assert_allclose(out[0, i], v[0, starts[i]:i + 1].mean(axis=0), atol=1e-14)
        np.testing.assert_allclose(lse[0, :, i], math.log(pos[i] + 1), atol=1e-14)


def test_dominant_key():
    rng = np.random.default_rng(9)
    S, H, D = 16, 1, 8
    q, k, v = (_rand((1, S, H, D), rng) for _ in range(3))
    q[0, S - 1, 0] = 0.0
    q[0, S - 1, 0, 0] = 200.0
    k[0, :, 0, 0] = 0.0
    k[0, 5, 0, 0] = 1.0                            # s_{S-1,5} = 200/sqrt(8) ~ 70.7, others 0
    out, _ = oracle.attention_forward(q, k, v, None)
    np.testing.assert_allclose(out[0, S - 1, 0], v[0, 5, 0], atol=1e-12)


# ----------------------------------------------------------------------------- invariants

def test_packed_row_equals_documents_alone():
    rng = np.random.default_rng(10)
    lens = [13, 1, 30, 20]
    S, H, D = sum(lens), 2, 8
    seg = np.repeat(np.arange(len(lens)), lens)[None]
    q, k, v, do = (_rand((1, S, H, D), rng) for _ in range(4))
    out, lse = oracle.attention_forward(q, k, v, seg)
    grads = oracle.attention_backward(q, k, v, do, seg)
    o = 0
    for L in lens:
        sl = slice(o, o + L)
        oo, ll = oracle.attention_forward(q[:, sl], k[:, sl], v[:, sl], None)
        np.testing.assert_allclose(out[:, sl], oo, atol=1e-13)
        np.testing.assert_allclose(lse[:, :, sl], ll, atol=1e-13)
        gg = oracle.attention_backward(q[:, sl], k[:, sl], v[:, sl], do[:, sl], None)
        for a, b in zip(grads, gg):
            np.testing.assert_allclose(a[:, sl], b, atol=1e-13)
        o += L


@pytest.mark.parametrize("bq,bk", [(1, 1), (7, 7), (64, 64), (128, 128), (200, 200), (5, 64), (64, 3)])
def test_blockwise_online_softmax_is_block_size_independent(bq, bk):
    rng = np.random.default_rng(11)
    S, H, D = 200, 2, 8
    seg = np.repeat([0, 1, 2, 3], [50, 1, 120, 29])
    q, k, v = (_rand((1, S, H, D), rng) * 2 for _ in range(3))
    out, lse = oracle.attention_forward(q, k, v, seg[None])
    for order in ("ascending", "descending"):
        bo, bl = BW.forward(q[0], k[0], v[0], seg, bq, bk, order)
        np.testing.assert_allclose(bo, out[0], atol=1e-12)
        np.testing.assert_allclose(bl, lse[0], atol=1e-12)


def test_shift_invariances_and_sum_rules():
    rng = np.random.default_rng(12)
    S, H, D = 60, 2, 8
    seg = np.repeat([0, 1, 2], [25, 5, 30])[None]
    q, k, v, do = (_rand((1, S, H, D), rng) for _ in range(4))
    out, lse = oracle.attention_forward(q, k, v, seg)
    c = rng.standard_normal(D)
    out_k, _ = oracle.attention_forward(q, k + c, v, seg)
    np.testing.assert_allclose(out_k, out, atol=1e-12)          # same c on every key
    out_v, _ = oracle.attention_forward(q, k, v + c, seg)
    np.testing.assert_allclose(out_v, out + c, atol=1e-12)      # rows of p sum to 1
    dq, dk, dv = oracle.attention_backward(q, k, v, do, seg)
    for d in range(3):
        m = seg[0] == d
        np.testing.assert_allclose(dk[0, m].sum(axis=0), 0.0, atol=1e-12)
        np.testing.assert_allclose(dv[0, m].sum(axis=0), do[0, m].sum(axis=0), atol=1e-12)


def test_large_scores_stay_finite():
    rng = np.random.default_rng(13)
    S, H, D = 64, 1, 16
    q, k, v, do = (_rand((1, S, H, D), rng) for _ in range(4))
    q *= 30.0
    out, lse = oracle.attention_forward(q, k, v, None)
    g = oracle.attention_backward(q, k, v, do, None)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    assert all(np.isfinite(x).all() for x in g)


def test_padding_rows_are_empty():
    rng = np.random.default_rng(14)
    S, H, D = 30, 1, 4
    seg = np.array([0] * 12 + [1] * 8 + [-1] * 10)[None]
    q, k, v, do = (_rand((1, S, H, D), rng) for _ in range(4))
    out, lse = oracle.attention_forward(q, k, v, seg)
    assert np.all(out[0, 20:] == 0) and np.all(np.isneginf(lse[0, :, 20:]))
    dq, dk, dv = oracle.attention_backward(q, k, v, do, seg)
    assert np.all(dq[0, 20:] == 0) and np.all(dk[0, 20:] == 0) and np.all(dv[0, 20:] == 0)
    o2, l2 = oracle.attention_forward(q[:, :20], k[:, :20], v[:, :20], seg[:, :20])
    np.testing.assert_allclose(out[:, :20], o2, atol=1e-14)


# ----------------------------------------------------------------------------- sampled modes

def test_sampled_rows_and_keys_match_full():
    rng = np.random.default_rng(15)
    B, S, H, D = 2, 300, 2, 8
    seg = np.stack([np.repeat([0, 1, 2], [100, 150, 50]), np.zeros(S, np.int64)])
    q, k, v, do = (_rand((B, S, H, D), rng) for _ in range(4))
    out, lse = oracle.attention_forward(q, k, v, seg)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, seg)
    rows = np.array([0, 1, 99, 100, 101, 249, 250, 299])
    for b in range(B):
        o, l = oracle.attention_forward_rows(q, k, v, seg, b, rows)
        np.testing.assert_allclose(o, out[b, rows], atol=1e-13)
        np.testing.assert_allclose(l, lse[b][:, rows], atol=1e-13)
        g = oracle.attention_backward_rows(q, k, v, do, seg, b, rows)
        np.testing.assert_allclose(g, dq[b, rows], atol=1e-13)
        for h in range(H):
            kk, vv = oracle.attention_key_grads(q, k, v, do, seg, b, h, rows)
            np.testing.assert_allclose(kk, dk[b, rows, h], atol=1e-13)
            np.testing.assert_allclose(vv, dv[b, rows, h], atol=1e-13)
            # the sum over queries split into disjoint query ranges adds up to the whole
            parts = [oracle.attention_key_grads(q, k, v, do, seg, b, h, rows, row_range=r)
                     for r in ((0, 70), (70, 260), (260, S))]
            np.testing.assert_allclose(sum(p[0] for p in parts), kk, atol=1e-13)
            np.testing.assert_allclose(sum(p[1] for p in parts), vv, atol=1e-13)
            # the row-block terms of the full backward add up to dq, dk, dv
            gk, gv = np.zeros((S, D)), np.zeros((S, D))
            for r in (np.arange(0, 37), np.arange(37, 180), np.arange(180, S)):
                g, j0, pk, pv = oracle.backward_row_block(q, k, v, do, seg, b, h, r)
                np.testing.assert_allclose(g, dq[b, r, h], atol=1e-13)
                gk[j0:j0 + len(pk)] += pk
                gv[j0:j0 + len(pv)] += pv
            np.testing.assert_allclose(gk, dk[b, :, h], atol=1e-13)
            np.testing.assert_allclose(gv, dv[b, :, h], atol=1e-13)


def test_credited_pairs_counts_the_visible_set():
    rng = np.random.default_rng(16)
    for _ in range(5):
        S = int(rng.integers(1, 40))
        seg = _random_segments(S, rng)[None]
        assert oracle.credited_pairs(seg) == int(oracle.visible_mask(seg[0], np.arange(S)).sum())


# ----------------------------------------------------------------------------- planted mistakes

def _planted(monkeypatch, kind):
    """Install a deliberately wrong oracle variant (CPU only)."""
    if kind == "strict_causal":
        def bad_mask(seg_row, rows):
            seg_row = np.asarray(seg_row); rows = np.asarray(rows)
            j = np.arange(seg_row.shape[0]); si = seg_row[rows][:, None]
            return (seg_row[None, :] == si) & (si >= 0) & (j[None, :] < rows[:, None]) | \
                   ((j[None, :] == rows[:, None]) & (rows[:, None] == 0))
        monkeypatch.setattr(OA, "visible_mask", bad_mask)
    elif kind == "no_segment":
        def bad_mask(seg_row, rows):
            seg_row = np.asarray(seg_row); rows = np.asarray(rows)
            j = np.arange(seg_row.shape[0])
            return (j[None, :] <= rows[:, None]) & (seg_row[rows][:, None] >= 0)
        monkeypatch.setattr(OA, "visible_mask", bad_mask)
    elif kind == "scale":
        orig = OA._rows_softmax
        monkeypatch.setattr(OA, "_rows_softmax", lambda q, k, s, r, scale: orig(q, k, s, r, scale * 1.01))


@pytest.mark.parametrize("kind", ["strict_causal", "no_segment", "scale"])
def test_planted_mistakes_are_caught(monkeypatch, kind):
    rng = np.random.default_rng(17)
    S, H, D = 12, 1, 4
    seg = np.repeat([0, 1], [5, 7])
    q, k, v = (_rand((1, S, H, D), rng) for _ in range(3))
    ref_o, _ = BF.forward(q[0].tolist(), k[0].tolist(), v[0].tolist(), seg.tolist())
    _planted(monkeypatch, kind)
    out, _ = oracle.attention_forward(q, k, v, seg[None])
    assert np.max(np.abs(out[0] - np.array(ref_o))) > 1e-6


def test_planted_gradient_mistake_is_caught():
    """A backward that forgets the delta term must disagree with finite differences."""
    rng = np.random.default_rng(18)
    S, H, D = 6, 1, 3
    seg = np.zeros((1, S), np.int64)
    q, k, v, do = (_rand((1, S, H, D), rng) for _ in range(4))
    scale = 1.0 / math.sqrt(D)
    dq_bad = np.zeros_like(q)
    for i in range(S):                                   # planted: ds = p * dp (no delta)
        p, _, j0, J = OA._rows_softmax(q[0, :, 0], k[0, :, 0], seg[0], np.array([i]), scale)
        dp = do[0, i, 0] @ v[0, j0:J, 0].T
        dq_bad[0, i, 0] = scale * ((p * dp) @ k[0, j0:J, 0])[0]
    h = 1e-6
    num = np.zeros_like(q)
    for idx in np.ndindex(q.shape):
        xp = q.copy(); xp[idx] += h
        xm = q.copy(); xm[idx] -= h
        num[idx] = (_loss(xp, k, v, do, seg) - _loss(xm, k, v, do, seg)) / (2 * h)
    assert np.linalg.norm(num - dq_bad) / np.linalg.norm(num) > 1e-3
    dq_good, _, _ = oracle.attention_backward(q, k, v, do, seg)
    assert np.linalg.norm(num - dq_good) / np.linalg.norm(num) < 1e-6
