"""Backward-pass parity: dq, dk, dv from the CUDA path against the float64 oracle.

Bar: relative L2 error <= 1e-2 per tensor over the checked elements. Small cases are
checked over every element; full-size workloads on 512 sampled query rows (dq) and
on sampled key rows of a few heads (dk, dv), which the oracle computes exactly from
the whole rows that see them.
"""

import numpy as np
import pytest
import torch

import blockwise_ringattention_causal_b300 as lwm
from blockwise_ringattention_causal_b300 import inputs as I
import oracle
from tests._oracle_pool import OraclePool
from tests._parity import GRAD_REL, f64, rel_l2

pytestmark = pytest.mark.gpu


def run_fwd_bwd(x, deterministic=True):
    out, lse, ws = lwm.forward(x["q"], x["k"], x["v"], x.get("seg"), x.get("pos"))
    dq, dk, dv = lwm.backward(x["q"], x["k"], x["v"], out, x["dout"], lse, x.get("seg"), x.get("pos"), ws,
                              fused=not deterministic)
    assert lwm.lwm_attn_check(ws) == 0
    return out, lse, dq, dk, dv


# both backward paths: separate dK/dV + dQ kernels (default) and the single kernel
PATHS = pytest.mark.parametrize("deterministic", [True, False], ids=["separate", "fused"])


def check_full(x, what, deterministic=True):
    _, _, dq, dk, dv = run_fwd_bwd(x, deterministic)
    seg = x["seg"].cpu().numpy() if x.get("seg") is not None else None
    refs = oracle.attention_backward(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["dout"]), seg)
    floor = 1e-3 * float(np.linalg.norm(f64(x["dout"])))
    errs = {n: rel_l2(f64(g), r, floor) for n, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), refs)}
    assert all(e <= GRAD_REL for e in errs.values()), f"{what}: {errs}"
    return errs


@PATHS
def test_packed_three_documents_s1k(cuda_device, deterministic):
    check_full(I.make_inputs(I.workload(1), cuda_device), "packed 300/424/300", deterministic)


@pytest.mark.parametrize("S,lengths", [
    (1, [[1]]), (127, [[127]]), (129, [[129]]), (300, [[100, 1, 199]]), (257, [[200, 30]]),
    (640, [[128, 128, 384]]), (500, [[7] * 70 + [10]]), (1000, [[1000]]),
])
@PATHS
def test_ragged_and_packed_shapes(cuda_device, S, lengths, deterministic):
    check_full(I.make_inputs(I.custom(1, S, 3, 128, lengths, seed=S), cuda_device), f"S={S}", deterministic)


@PATHS
def test_batch_rows_with_padding(cuda_device, deterministic):
    x = I.make_inputs(I.custom(3, 700, 2, 128, [[700], [50, 650], [300, 300, 64]], seed=5), cuda_device)
    check_full(x, "B=3", deterministic)
    _, _, dq, dk, dv = run_fwd_bwd(x, deterministic)
    for g in (dq, dk, dv):
        assert torch.all(g[2, 664:] == 0)


def test_separate_path_is_deterministic(cuda_device):
    x = I.make_inputs(I.custom(1, 3000, 4, 128, [[1000, 2000]], seed=8), cuda_device)
    a = run_fwd_bwd(x, deterministic=True)
    b = run_fwd_bwd(x, deterministic=True)
    for u, w in zip(a, b):
        assert torch.equal(u, w)


def test_fused_path_repeats_dk_dv_exactly(cuda_device):
    """dk and dv of the single-kernel path are bitwise reproducible; dq is summed in fp32
    in a scheduling-dependent order, so two runs agree to fp32 rounding before the bf16
    conversion: at most one bf16 unit in the last place apart."""
    x = I.make_inputs(I.custom(1, 3000, 4, 128, [[1000, 2000]], seed=8), cuda_device)
    a = run_fwd_bwd(x, deterministic=False)
    b = run_fwd_bwd(x, deterministic=False)
    for u, w in zip(a[:2] + a[3:], b[:2] + b[3:]):
        assert torch.equal(u, w)
    dq_a, dq_b = a[2].float(), b[2].float()
    bound = torch.maximum(dq_a.abs(), dq_b.abs()) * 2.0 ** -7 + 1e-5 * float(dq_a.abs().max())
    assert torch.all((dq_a - dq_b).abs() <= bound)


def test_fused_and_separate_paths_agree(cuda_device):
    x = I.make_inputs(I.custom(2, 1500, 3, 128, [[700, 800], [1500]], seed=11), cuda_device)
    f = run_fwd_bwd(x, deterministic=False)
    d = run_fwd_bwd(x, deterministic=True)
    for name, g, h in zip(("dq", "dk", "dv"), f[2:], d[2:]):
        assert rel_l2(f64(g), f64(h)) <= 5e-3, name


@PATHS
def test_large_scores_stay_finite(cuda_device, deterministic):
    x = I.make_inputs(I.custom(1, 512, 2, 128, [[512]], seed=9), cuda_device)
    x["q"] = (x["q"].float() * 30).to(torch.bfloat16)
    _, _, dq, dk, dv = run_fwd_bwd(x, deterministic)
    for g in (dq, dk, dv):
        assert torch.isfinite(g.float()).all()


def _sampled_bwd(config, cuda_device, key_heads=(0, 17), deterministic=True):
    w = I.workload(config)
    x = I.make_inputs(w, cuda_device)
    _, _, dq, dk, dv = run_fwd_bwd(x, deterministic)
    rows = I.sample_rows(w.S)
    keys = I.sample_rows(w.S, seed=2)
    seg = x["seg"].cpu().numpy()
    got, ref = [], []
    for b in range(w.B):
        for h in range(w.H):
            q, k, v, do = (x[n][b:b + 1, :, h:h + 1].float().cpu().numpy() for n in ("q", "k", "v", "dout"))
            r = oracle.attention_backward_rows(q, k, v, do, seg[b:b + 1], 0, rows)
            got.append(f64(dq[b, rows, h])); ref.append(r[:, 0])
    e_dq = rel_l2(np.stack(got), np.stack(ref))
    gk, gv, rk, rv = [], [], [], []
    for h in key_heads:
        q, k, v, do = (x[n][0:1, :, h:h + 1].float().cpu().numpy() for n in ("q", "k", "v", "dout"))
        kk, vv = oracle.attention_key_grads(q, k, v, do, seg[0:1], 0, 0, keys)
        gk.append(f64(dk[0, keys, h])); rk.append(kk)
        gv.append(f64(dv[0, keys, h])); rv.append(vv)
    e_dk = rel_l2(np.stack(gk), np.stack(rk))
    e_dv = rel_l2(np.stack(gv), np.stack(rv))
    assert max(e_dq, e_dk, e_dv) <= GRAD_REL, f"config {config}: dq {e_dq:.2e} dk {e_dk:.2e} dv {e_dv:.2e}"


@PATHS
def test_causal_s32k_sampled(cuda_device, deterministic):
    _sampled_bwd(2, cuda_device, deterministic=deterministic)


def test_packed_mixed_s64k_sampled(cuda_device):
    _sampled_bwd(3, cuda_device, key_heads=(5,))


def test_video_s256k_sampled_and_invariants(cuda_device):
    """256K tokens (1024 frames of 256 tokens with a shared per-frame offset).

    dq on 512 sampled query rows of a subset of heads (exact from each row alone); dk, dv
    on the last 256 keys of two heads and on 256 keys of the first four frames of two
    heads (exact from every row that sees them); and on every head the identities that hold at any size: sum_j dv_j = sum_i dout_i (each row's
    probabilities sum to 1) and sum_j dk_j = 0 (each row's dS sums to 0).
    """
    w = I.workload(4)
    x = I.make_inputs(w, cuda_device)
    _, _, dq, dk, dv = run_fwd_bwd(x)
    seg = x["seg"].cpu().numpy()
    rows = I.sample_rows(w.S)
    got, ref = [], []
    for h in (0, 13, 31):
        q, k, v, do = (x[n][0:1, :, h:h + 1].float().cpu().numpy() for n in ("q", "k", "v", "dout"))
        for c in range(0, len(rows), 64):
            r = rows[c:c + 64]
            ref.append(oracle.attention_backward_rows(q, k, v, do, seg[0:1], 0, r)[:, 0])
            got.append(f64(dq[0, r, h]))
    e_dq = rel_l2(np.concatenate(got), np.concatenate(ref))
    keys = np.arange(w.S - 256, w.S)
    gk, gv, rk, rv = [], [], [], []
    for h in (4, 22):
        q, k, v, do = (x[n][0:1, :, h:h + 1].float().cpu().numpy() for n in ("q", "k", "v", "dout"))
        kk, vv = oracle.attention_key_grads(q, k, v, do, seg[0:1], 0, 0, keys)
        gk.append(f64(dk[0, keys, h])); rk.append(kk)
        gv.append(f64(dv[0, keys, h])); rv.append(vv)
    e_dk = rel_l2(np.concatenate(gk), np.concatenate(rk))
    e_dv = rel_l2(np.concatenate(gv), np.concatenate(rv))
    assert max(e_dq, e_dk, e_dv) <= GRAD_REL, f"dq {e_dq:.2e} dk {e_dk:.2e} dv {e_dv:.2e}"
    # 256 early keys (frames 0-3) of two heads: each column sums over ~262K queries, the
    # long accumulations of the persistent dK/dV kernel; the oracle forms every row
    early = np.sort(np.random.default_rng(4).choice(4 * I.FRAME_TOKENS, 256, replace=False))
    heads = (4, 22)
    tensors = {n: x[n][:, :, list(heads)].float().cpu().numpy() for n in ("q", "k", "v", "dout")}
    with OraclePool(tensors, seg) as pool:
        ref = pool.key_grads(0, [0, 1], early)
    gk = np.stack([f64(dk[0, early, h]) for h in heads])
    gv = np.stack([f64(dv[0, early, h]) for h in heads])
    e_dk = rel_l2(gk, np.stack([ref[i][0] for i in range(2)]))
    e_dv = rel_l2(gv, np.stack([ref[i][1] for i in range(2)]))
    assert max(e_dk, e_dv) <= GRAD_REL, f"early keys: dk {e_dk:.2e} dv {e_dv:.2e}"
    # identities over all heads, in float64 on the device
    sum_dv = dv[0].double().sum(dim=0)            # [H, D]
    sum_do = x["dout"][0].double().sum(dim=0)
    assert float((sum_dv - sum_do).norm() / sum_do.norm()) <= GRAD_REL
    sum_dk = dk[0].double().sum(dim=0)
    assert float(sum_dk.norm() / dk[0].double().norm()) <= GRAD_REL
