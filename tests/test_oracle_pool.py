"""The process-pool runner of the oracle (used by the full-size GPU parity tests)
returns exactly what the plain oracle functions return (CPU only)."""

import numpy as np

import oracle
from tests._oracle_pool import OraclePool, _row_groups


def test_row_groups_cover_the_rows_in_order():
    seg = np.repeat([0, 1, 2, -1], [300, 1, 500, 99])
    g = _row_groups(seg, 5)
    assert g[0][0] == 0 and g[-1][1] == len(seg)
    assert all(a[1] == b[0] for a, b in zip(g[:-1], g[1:]))


def test_pool_matches_the_oracle():
    rng = np.random.default_rng(3)
    B, S, H, D = 2, 700, 2, 16
    seg = np.stack([np.repeat([0, 1, 2, -1], [300, 1, 350, 49]), np.zeros(S, np.int64)])
    x = {n: rng.standard_normal((B, S, H, D)).astype(np.float32) for n in ("q", "k", "v", "dout")}
    ref_o, ref_l = oracle.attention_forward(x["q"], x["k"], x["v"], seg)
    ref_g = oracle.attention_backward(x["q"], x["k"], x["v"], x["dout"], seg)
    with OraclePool(x, seg, workers=2) as pool:
        o, l = pool.forward()
        g = pool.backward()
        keys = np.array([0, 5, 299, 300, 301, 640, 699])
        kg = pool.key_grads(1, [0, 1], keys, per_head=3)
        kg0 = pool.key_grads(0, [1], keys, per_head=2)
    np.testing.assert_allclose(o, ref_o, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(l), np.isneginf(ref_l))
    fin = np.isfinite(ref_l)
    np.testing.assert_allclose(l[fin], ref_l[fin], atol=1e-12)
    for a, r in zip(g, ref_g):
        np.testing.assert_allclose(a, r, atol=1e-12)
    for h in (0, 1):
        np.testing.assert_allclose(kg[h][0], ref_g[1][1, keys, h], atol=1e-12)
        np.testing.assert_allclose(kg[h][1], ref_g[2][1, keys, h], atol=1e-12)
    np.testing.assert_allclose(kg0[1][0], ref_g[1][0, keys, 1], atol=1e-12)
    np.testing.assert_allclose(kg0[1][1], ref_g[2][0, keys, 1], atol=1e-12)
