"""Pins for the RoPE oracle (oracle/rope.py), against things other than itself (CPU).

  * a worked example derived by hand from the definition (tests/golden/rope_worked_example_d4.json);
  * what rotations must satisfy: the inverse undoes the rotation, norms are kept,
    position 0 is the identity;
  * what RoPE is for: shifting every position of a document by the same amount leaves
    the attention output unchanged (scores depend only on relative positions);
  * central finite differences of L = sum(dO * O) for the gradients with respect to
    the unrotated q and k;
  * bf16 rounding against torch's float32 -> bfloat16 conversion (a library routine);
  * planted mistakes (the rotate-half pairing, a wrong sign, a wrong frequency
    exponent) fail the worked example.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import rope as R

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "rope_worked_example_d4.json")


def _golden():
    g = json.load(open(GOLDEN))
    ev = lambda e: float(eval(e, {"__builtins__": {}}, {"cos": math.cos, "sin": math.sin}))  # noqa: E731
    x = np.array(g["x"], np.float64)[None, :, None, :]
    pos = np.array(g["pos"])[None]
    rot = np.array([[ev(e) for e in r] for r in g["rotated"]])
    inv = np.array([[ev(e) for e in r] for r in g["inverse"]])
    return x, pos, g["theta"], rot, inv


def test_worked_example():
    x, pos, theta, rot, inv = _golden()
    np.testing.assert_allclose(R.rope_rotate(x, pos, theta)[0, :, 0], rot, atol=1e-14)
    np.testing.assert_allclose(R.rope_rotate(x, pos, theta, inverse=True)[0, :, 0], inv, atol=1e-14)


@pytest.mark.parametrize("kind", ["rotate_half", "sign", "exponent"])
def test_planted_mistakes_fail_the_worked_example(kind):
    x, pos, theta, rot, _ = _golden()
    D = x.shape[-1]
    ang = R.rope_angles(pos, theta, D)
    c, s = np.cos(ang)[:, :, None, :], np.sin(ang)[:, :, None, :]
    y = np.empty_like(x)
    if kind == "rotate_half":            # pairs (m, m + D/2) instead of (2m, 2m+1)
        a, b = x[..., : D // 2], x[..., D // 2:]
        y[..., : D // 2], y[..., D // 2:] = a * c - b * s, a * s + b * c
    elif kind == "sign":
        a, b = x[..., 0::2], x[..., 1::2]
        y[..., 0::2], y[..., 1::2] = a * c + b * s, -a * s + b * c
    else:                                # theta^(-m/D)
        ang2 = np.asarray(pos, np.float64)[..., None] * np.power(theta, -np.arange(D // 2) / D)
        c2, s2 = np.cos(ang2)[:, :, None, :], np.sin(ang2)[:, :, None, :]
        a, b = x[..., 0::2], x[..., 1::2]
        y[..., 0::2], y[..., 1::2] = a * c2 - b * s2, a * s2 + b * c2
    assert np.max(np.abs(y[0, :, 0] - rot)) > 1e-3


def test_inverse_norm_and_identity_at_position_zero():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((2, 50, 3, 128))
    pos = rng.integers(0, 1 << 20, size=(2, 50))
    pos[0, 0] = 0
    for theta in (1e4, 1e6, 5e7):
        y = R.rope_rotate(x, pos, theta)
        np.testing.assert_allclose(R.rope_rotate(y, pos, theta, inverse=True), x, atol=1e-12)
        np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)
        np.testing.assert_allclose(y[0, 0], x[0, 0], atol=0)


def test_shifting_a_documents_positions_leaves_attention_unchanged():
    rng = np.random.default_rng(1)
    S, H, D = 60, 2, 16
    q, k, v = (rng.standard_normal((1, S, H, D)) for _ in range(3))
    seg = np.repeat([0, 1, 2], [20, 25, 15])[None]
    pos = np.concatenate([np.arange(20), np.arange(25), np.arange(15)])[None]
    shifted = pos + np.repeat([1000, 37, 123456], [20, 25, 15])[None]
    for theta in (1e4, 1e6, 5e7):
        o1, l1 = R.attention_forward_rope(q, k, v, seg, pos, theta, bf16_inputs=False)
        o2, l2 = R.attention_forward_rope(q, k, v, seg, shifted, theta, bf16_inputs=False)
        np.testing.assert_allclose(o2, o1, atol=1e-9)
        np.testing.assert_allclose(l2, l1, atol=1e-9)
    # and it does change when only some tokens of a document move
    bad = pos.copy()
    bad[0, 5] += 3
    o3, _ = R.attention_forward_rope(q, k, v, seg, bad, 1e4, bf16_inputs=False)
    assert np.max(np.abs(o3 - o1)) > 1e-6


def _loss(q, k, v, do, seg, pos, theta):
    out, _ = R.attention_forward_rope(q, k, v, seg, pos, theta, bf16_inputs=False)
    return float(np.sum(out * do))


def test_finite_differences():
    rng = np.random.default_rng(2)
    S, H, D = 7, 1, 4
    q, k, v, do = (rng.standard_normal((1, S, H, D)) for _ in range(4))
    seg = np.repeat([0, 1], [3, 4])[None]
    pos = np.array([[0, 1, 2, 0, 1, 2, 3]]) * 3
    theta = 100.0
    gq, gk, gv = R.attention_backward_rope(q, k, v, do, seg, pos, theta, bf16_inputs=False)
    h = 1e-6
    for x, g in ((q, gq), (k, gk), (v, gv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            args = [q, k, v]
            which = 0 if x is q else (1 if x is k else 2)
            ap, am = list(args), list(args)
            ap[which], am[which] = xp, xm
            num[idx] = (_loss(*ap, do, seg, pos, theta) - _loss(*am, do, seg, pos, theta)) / (2 * h)
        assert np.linalg.norm(num - g) / np.linalg.norm(num) < 1e-6


def test_round_bf16_matches_torch():
    rng = np.random.default_rng(3)
    x32 = (rng.standard_normal(100000) * np.exp(rng.uniform(-20, 20, 100000))).astype(np.float32)
    # exact ties: 8 significant bits plus a half unit in the last place
    ties = (np.arange(128, 256, dtype=np.float32) + np.float32(0.5)) * np.float32(2.0 ** -7)
    x32 = np.concatenate([x32, ties, -ties, np.float32([0.0, 1.0, -3.0])])
    ref = torch.from_numpy(x32).to(torch.bfloat16).float().numpy().astype(np.float64)
    np.testing.assert_array_equal(R.round_bf16(x32.astype(np.float64)), ref)


def test_exported_from_the_oracle_package():
    assert oracle.rope_rotate is R.rope_rotate
    assert oracle.attention_backward_rope is R.attention_backward_rope
