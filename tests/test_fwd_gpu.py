"""Forward-pass parity: the CUDA path (through the C ABI) against the float64 oracle.

Small cases are compared element by element over every output; the full-size
workloads are compared on 512 sampled query rows (all heads) that the oracle
computes one by one.
"""

import numpy as np
import pytest
import torch

import blockwise_ringattention_causal_b300 as lwm
from blockwise_ringattention_causal_b300 import inputs as I
import oracle
from tests._parity import assert_fwd, f64

pytestmark = pytest.mark.gpu


def run_fwd(x, kv_chunks=1):
    B, S, H, D = x["q"].shape
    ws = lwm.new_workspace(B, S, H, D, x["q"].device, forward_only=True)
    out, lse, ws = lwm.forward(x["q"], x["k"], x["v"], x.get("seg"), x.get("pos"), kv_chunks=kv_chunks, workspace=ws)
    assert lwm.lwm_attn_check(ws) == 0
    return out, lse


def full_ref(x):
    seg = x["seg"].cpu().numpy() if x.get("seg") is not None else None
    return oracle.attention_forward(f64(x["q"]), f64(x["k"]), f64(x["v"]), seg)


def test_packed_three_documents_s1k(cuda_device):
    x = I.make_inputs(I.workload(1), cuda_device, with_dout=False)
    out, lse = run_fwd(x)
    ref_o, ref_l = full_ref(x)
    assert_fwd(f64(out), f64(lse), ref_o, ref_l, "packed 300/424/300")


@pytest.mark.parametrize("S,lengths", [
    (1, [[1]]), (127, [[127]]), (129, [[129]]), (300, [[100, 1, 199]]), (257, [[200, 30]]),
    (1000, [[1000]]), (640, [[128, 128, 384]]), (500, [[7] * 70 + [10]]),
])
def test_ragged_and_packed_shapes(cuda_device, S, lengths):
    w = I.custom(1, S, 3, 128, lengths, seed=S)
    x = I.make_inputs(w, cuda_device, with_dout=False)
    out, lse = run_fwd(x)
    ref_o, ref_l = full_ref(x)
    assert_fwd(f64(out), f64(lse), ref_o, ref_l, f"S={S}", bf16_bound=True)


def test_batch_rows_with_different_packings(cuda_device):
    w = I.custom(3, 700, 2, 128, [[700], [50, 650], [300, 300, 64]], seed=5)   # row 2 ends in padding
    x = I.make_inputs(w, cuda_device, with_dout=False)
    assert (x["seg"][2, 664:] == -1).all()
    out, lse = run_fwd(x)
    ref_o, ref_l = full_ref(x)
    assert_fwd(f64(out), f64(lse), ref_o, ref_l, "B=3", bf16_bound=True)
    assert torch.all(out[2, 664:] == 0)


def test_pos_and_seg_defaults(cuda_device):
    w = I.custom(1, 600, 2, 128, [[200, 400]], seed=6)
    x = I.make_inputs(w, cuda_device, with_dout=False)
    o1, l1 = run_fwd(x)
    o2, l2 = run_fwd({**x, "pos": None})                 # pos derived from seg
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    w1 = I.custom(1, 600, 2, 128, None, seed=6)
    x1 = I.make_inputs(w1, cuda_device, with_dout=False)
    o3, l3 = run_fwd({**x1, "seg": None, "pos": None})   # one document per row
    ref_o, ref_l = full_ref({**x1, "seg": None})
    assert_fwd(f64(o3), f64(l3), ref_o, ref_l, "seg=None")


@pytest.mark.parametrize("chunks", [2, 3, 8])
def test_ring_order_is_order_independent(cuda_device, chunks):
    w = I.custom(1, 2000, 2, 128, [[900, 1100]], seed=7)
    x = I.make_inputs(w, cuda_device, with_dout=False)
    out, lse = run_fwd(x, kv_chunks=chunks)
    ref_o, ref_l = full_ref(x)
    assert_fwd(f64(out), f64(lse), ref_o, ref_l, f"ring {chunks}")


def test_forward_is_deterministic(cuda_device):
    x = I.make_inputs(I.custom(1, 3000, 4, 128, [[1000, 2000]], seed=8), cuda_device, with_dout=False)
    o1, l1 = run_fwd(x)
    o2, l2 = run_fwd(x)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_large_scores_stay_finite(cuda_device):
    x = I.make_inputs(I.custom(1, 512, 2, 128, [[512]], seed=9), cuda_device, with_dout=False)
    x["q"] = (x["q"].float() * 30).to(torch.bfloat16)
    out, lse = run_fwd(x)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    ref_o, ref_l = full_ref(x)
    assert_fwd(f64(out), f64(lse), ref_o, ref_l, "q x 30", bf16_bound=True)


def test_bad_segments_are_reported(cuda_device):
    w = I.custom(1, 256, 1, 128, [[100, 156]], seed=10)
    x = I.make_inputs(w, cuda_device, with_dout=False)
    bad_seg = x["seg"].clone()
    bad_seg[0, 200:] = 0                                  # id goes back down: not contiguous runs
    _, _, ws = lwm.forward(x["q"], x["k"], x["v"], bad_seg, None)
    assert lwm.lwm_attn_check(ws) == 4
    bad_pos = x["pos"].clone()
    bad_pos[0, 150] += 1                                  # pos inconsistent with seg
    _, _, ws = lwm.forward(x["q"], x["k"], x["v"], x["seg"], bad_pos)
    assert lwm.lwm_attn_check(ws) == 4
    assert lwm.lwm_attn_check(ws) == 0                    # the check clears the word


def _sampled(config, cuda_device):
    w = I.workload(config)
    x = I.make_inputs(w, cuda_device, with_dout=False)
    out, lse = run_fwd(x, kv_chunks=w.kv_chunks)
    rows = I.sample_rows(w.S)
    seg = x["seg"].cpu().numpy()
    outs, refs = [], []
    for b in range(w.B):
        for h in range(w.H):
            q, k, v = (x[n][b:b + 1, :, h:h + 1].float().cpu().numpy() for n in ("q", "k", "v"))
            ref_o, ref_l = oracle.attention_forward_rows(q, k, v, seg[b:b + 1], 0, rows)
            outs.append((f64(out[b, rows, h]), f64(lse[b, h, rows])))
            refs.append((ref_o[:, 0], ref_l[0]))
    got_o = np.stack([o for o, _ in outs]); got_l = np.stack([l for _, l in outs])
    ref_o = np.stack([o for o, _ in refs]); ref_l = np.stack([l for _, l in refs])
    assert_fwd(got_o, got_l, ref_o, ref_l, f"config {config}")


def test_causal_s32k_sampled_rows(cuda_device):
    _sampled(2, cuda_device)


def test_packed_mixed_s64k_sampled_rows(cuda_device):
    _sampled(3, cuda_device)


# ----------------------------------------------------------------------------- 256K and 1M tokens
# The whole-row oracle is exact but costs O(rows x S x D) host flops per head, so at
# S >= 256K it runs on 512 sampled query rows of a spread subset of heads.
SAMPLED_HEADS_256K = (0, 9, 18, 27)
SAMPLED_HEADS_1M = (0, 10, 21, 31)


def _sampled_heads(w, x, out, lse, heads, rows_per_call):
    rows = I.sample_rows(w.S)
    seg = x["seg"].cpu().numpy()
    got_o, got_l, ref_o, ref_l = [], [], [], []
    for h in heads:
        q, k, v = (x[n][0:1, :, h:h + 1].float().cpu().numpy() for n in ("q", "k", "v"))
        for c in range(0, len(rows), rows_per_call):
            r = rows[c:c + rows_per_call]
            o, l = oracle.attention_forward_rows(q, k, v, seg[0:1], 0, r)
            ref_o.append(o[:, 0]); ref_l.append(l[0])
            got_o.append(f64(out[0, r, h])); got_l.append(f64(lse[0, h, r]))
    assert_fwd(np.concatenate(got_o), np.concatenate(got_l), np.concatenate(ref_o), np.concatenate(ref_l),
               f"{w.name} heads {heads}")


def test_video_s256k_sampled_rows(cuda_device):
    w = I.workload(4)
    x = I.make_inputs(w, cuda_device, with_dout=False)
    out, lse = run_fwd(x, kv_chunks=w.kv_chunks)
    _sampled_heads(w, x, out, lse, SAMPLED_HEADS_256K, 64)


def test_ring_order_s1m_sampled_rows(cuda_device):
    """1M tokens in one launch, key/value chunks visited in ring order (8 chunks)."""
    w = I.workload(5)
    assert w.kv_chunks == 8 and not w.backward
    x = I.make_inputs(w, cuda_device, with_dout=False)
    out, lse = run_fwd(x, kv_chunks=w.kv_chunks)
    assert torch.isfinite(lse).all()
    _sampled_heads(w, x, out, lse, SAMPLED_HEADS_1M, 16)
