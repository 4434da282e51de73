"""RoPE on q and k (lwm_attn_rope) against the float64 oracle (oracle/rope.py).

  * The rotation itself, every element, against the oracle's rotation rounded to bf16:
    the kernel rotates in fp32, so an element may land one bf16 unit (plus the fp32
    error of the pair, within 2^-20 of its magnitude) away from the float64 result, where that
    result lies within fp32 rounding of a rounding boundary; rarely (<= 1e-3).
  * Attention with RoPE (rotate, attention on the rotated q and k, rotate dq and dk
    back): the packed 1K workload on every element, the 32K workload on 512 sampled
    query rows of every head and on sampled keys of two heads, at theta = 1e6 (LWM's
    32K stage) and 5e7 (its 1M stage).
"""

import numpy as np
import pytest
import torch

import blockwise_ringattention_causal_b300 as lwm
from blockwise_ringattention_causal_b300 import inputs as I
import oracle
from tests._oracle_pool import OraclePool
from tests._parity import GRAD_REL, assert_fwd, f64, rel_l2

pytestmark = pytest.mark.gpu

THETAS = (1e6, 5e7)
KEY_HEADS = (3, 28)


def _check_rotation(x, pos, theta, inverse, what):
    """Every element against the float64 rotation rounded to bf16. The kernel rotates in
    fp32: y32 = x0 c - x1 s (or x0 s + x1 c) is within 2^-20 (|x0| + |x1|) of the float64
    y (the reduced angle rounded to fp32, sin/cos, two products), and each side then
    rounds to bf16, so |out - ref| <= 2^-20 (|x0| + |x1|) plus a bf16 unit of out or ref.
    Elements that differ at all stay rare (<= 1e-3)."""
    out, _ = lwm.rope(x, None, pos, theta, inverse=inverse)
    p = pos.cpu().numpy() if pos is not None else np.broadcast_to(np.arange(x.shape[1]), x.shape[:2])
    xf = f64(x)
    ref = oracle.round_bf16(oracle.rope_rotate(xf, p, theta, inverse=inverse))
    got = f64(out)
    mag = np.repeat(np.abs(xf[..., 0::2]) + np.abs(xf[..., 1::2]), 2, axis=-1)
    ulp = lambda t: np.ldexp(1.0, np.frexp(np.abs(t))[1] - 8)   # noqa: E731  bf16 spacing at t
    bound = 2.0 ** -20 * mag + np.maximum(ulp(ref), ulp(got))
    excess = np.abs(got - ref) - bound
    assert excess.max() <= 0, f"{what}: bound exceeded by {excess.max():.3e}"
    assert (got != ref).mean() <= 1e-3, f"{what}: {(got != ref).mean():.2e} of the elements differ"


@pytest.mark.parametrize("theta", THETAS)
def test_rotation_every_element(cuda_device, theta):
    x = I.make_inputs(I.workload(1), cuda_device, with_dout=False)
    for inverse in (False, True):
        _check_rotation(x["q"], x["pos"], theta, inverse, f"packed 1K theta {theta:g} inverse {inverse}")
    w = I.workload(2)
    x = I.make_inputs(w, cuda_device, with_dout=False)
    _check_rotation(x["k"], x["pos"], theta, False, f"32K theta {theta:g}")
    # positions near 2^20 (the 1M stage): angles up to 1e6 rad
    big = I.custom(2, 4096, 2, 128, None, seed=3)
    xb = I.make_inputs(big, cuda_device, with_dout=False)
    pos = (torch.arange(4096, dtype=torch.int32, device=cuda_device) + (1 << 20) - 4096).repeat(2, 1).contiguous()
    _check_rotation(xb["q"], pos, theta, False, f"positions near 1M theta {theta:g}")
    _check_rotation(xb["q"], None, theta, True, f"pos = NULL theta {theta:g}")


def test_both_tensors_and_in_place(cuda_device):
    x = I.make_inputs(I.workload(1), cuda_device, with_dout=False)
    qr, kr = lwm.rope(x["q"], x["k"], x["pos"], 1e6)
    q2 = x["q"].clone()
    lwm.lwm_attn_rope(q2, None, x["pos"], 1e6, q2, None)
    assert torch.equal(q2, qr)
    k_only, _ = lwm.rope(x["k"], None, x["pos"], 1e6)
    assert torch.equal(k_only, kr)
    back, _ = lwm.rope(qr, None, x["pos"], 1e6, inverse=True)
    assert rel_l2(f64(back), f64(x["q"])) < 1e-2


def _rope_fwd_bwd(x, theta):
    qr, kr = lwm.rope(x["q"], x["k"], x["pos"], theta)
    out, lse, ws = lwm.forward(qr, kr, x["v"], x["seg"], x["pos"])
    dqr, dkr, dv = lwm.backward(qr, kr, x["v"], out, x["dout"], lse, x["seg"], x["pos"], ws)
    assert lwm.lwm_attn_check(ws) == 0
    dq, dk = lwm.rope(dqr, dkr, x["pos"], theta, inverse=True)
    return out, lse, dq, dk, dv


@pytest.mark.parametrize("theta", THETAS)
def test_attention_with_rope_packed_1k(cuda_device, theta):
    x = I.make_inputs(I.workload(1), cuda_device)
    out, lse, dq, dk, dv = _rope_fwd_bwd(x, theta)
    seg, pos = x["seg"].cpu().numpy(), x["pos"].cpu().numpy()
    q, k, v, do = (f64(x[n]) for n in ("q", "k", "v", "dout"))
    ref_o, ref_l = oracle.attention_forward_rope(q, k, v, seg, pos, theta)
    assert_fwd(f64(out), f64(lse), ref_o, ref_l, f"rope {theta:g}")
    refs = oracle.attention_backward_rope(q, k, v, do, seg, pos, theta)
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        assert rel_l2(f64(g), r) <= GRAD_REL, name


@pytest.mark.parametrize("theta", THETAS)
def test_attention_with_rope_s32k_sampled(cuda_device, theta):
    w = I.workload(2)
    x = I.make_inputs(w, cuda_device)
    out, lse, dq, dk, dv = _rope_fwd_bwd(x, theta)
    seg, pos = x["seg"].cpu().numpy(), x["pos"].cpu().numpy()
    rows = I.sample_rows(w.S)
    got_o, got_l, ref_o, ref_l, got_q, ref_q = [], [], [], [], [], []
    rotated = {}
    for h in range(w.H):
        q, k, v, do = (x[n][:, :, h:h + 1].float().cpu().numpy() for n in ("q", "k", "v", "dout"))
        qr = oracle.round_bf16(oracle.rope_rotate(q, pos, theta))
        kr = oracle.round_bf16(oracle.rope_rotate(k, pos, theta))
        o, l = oracle.attention_forward_rows(qr, kr, v, seg, 0, rows)
        ref_o.append(o[:, 0]); ref_l.append(l[0])
        got_o.append(f64(out[0, rows, h])); got_l.append(f64(lse[0, h, rows]))
        g = oracle.attention_backward_rows(qr, kr, v, do, seg, 0, rows)       # [R, 1, D], rotated frame
        ref_q.append(oracle.rope_rotate(g[None], pos[:, rows], theta, inverse=True)[0, :, 0])
        got_q.append(f64(dq[0, rows, h]))
        if h in KEY_HEADS:
            rotated[h] = (qr, kr, v, do)
    assert_fwd(np.stack(got_o), np.stack(got_l), np.stack(ref_o), np.stack(ref_l), f"rope 32K {theta:g}")
    assert rel_l2(np.stack(got_q), np.stack(ref_q)) <= GRAD_REL
    # dk, dv on sampled keys of two heads (every query that sees them), in the rotated
    # frame from the oracle, then rotated back
    keys = I.sample_rows(w.S, seed=2)
    tensors = {n: np.concatenate([rotated[h][i] for h in KEY_HEADS], axis=2).astype(np.float32)
               for i, n in enumerate(("q", "k", "v", "dout"))}
    with OraclePool(tensors, seg) as pool:
        ref = pool.key_grads(0, list(range(len(KEY_HEADS))), keys)
    for i, h in enumerate(KEY_HEADS):
        kk = oracle.rope_rotate(ref[i][0][None, :, None, :], pos[:, keys], theta, inverse=True)[0, :, 0]
        assert rel_l2(f64(dk[0, keys, h]), kk) <= GRAD_REL, f"dk head {h}"
        assert rel_l2(f64(dv[0, keys, h]), ref[i][1]) <= GRAD_REL, f"dv head {h}"
