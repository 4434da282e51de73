"""Decoding against a key/value cache (lwm_attn_decode) against the float64 oracle.

Query t of row b sits at position P = kv_len[b] - T + t of its row and attends to keys
0 .. P: the oracle's forward rows at those positions (the same definition as the
prefill path). Cache entries past kv_len are filled with NaN, so any read of them
shows. Bar: the forward one (max |out - o| <= 1e-2, mean <= 1e-3, lse <= 1e-3).
"""

import numpy as np
import pytest
import torch

import blockwise_ringattention_causal_b300 as lwm
from blockwise_ringattention_causal_b300 import inputs as I
import oracle
from tests._parity import assert_fwd, f64

pytestmark = pytest.mark.gpu


def _case(B, S_max, H, T, kv_len, cuda_device, seed):
    x = I.make_inputs(I.custom(B, S_max, H, 128, None, seed=seed), cuda_device, with_dout=False)
    q_full, k, v = x["q"], x["k"].clone(), x["v"].clone()
    for b, L in enumerate(kv_len):
        k[b, L:] = float("nan")
        v[b, L:] = float("nan")
    pos = torch.stack([torch.arange(L - T, L) for L in kv_len]).to(cuda_device)   # [B, T]
    q = torch.stack([q_full[b, pos[b]] for b in range(B)]).contiguous()              # [B, T, H, D]
    lens = torch.tensor(kv_len, dtype=torch.int32, device=cuda_device)
    return q_full, q, k, v, lens, pos.cpu().numpy()


def _reference(q_full, k, v, pos):
    B, T = pos.shape
    H = q_full.shape[2]
    ref_o = np.zeros((B, T, H, 128))
    ref_l = np.zeros((B, H, T))
    qf, kf, vf = f64(q_full), np.nan_to_num(f64(k)), np.nan_to_num(f64(v))
    for b in range(B):
        o, l = oracle.attention_forward_rows(qf, kf, vf, None, b, pos[b])
        ref_o[b], ref_l[b] = o, l
    return ref_o, ref_l


@pytest.mark.parametrize("T", [1, 2, 3, 4])
def test_ragged_rows_every_element(cuda_device, T):
    B, S_max, H = 3, 3000, 20                      # 20 heads: a full and a partial group of 16
    kv_len = [3000, 1537, T]
    q_full, q, k, v, lens, pos = _case(B, S_max, H, T, kv_len, cuda_device, seed=T)
    out, lse, ws = lwm.decode(q, k, v, lens)
    assert lwm.lwm_attn_check(ws) == 0
    ref_o, ref_l = _reference(q_full, k, v, pos)
    assert_fwd(f64(out), f64(lse), ref_o, ref_l, f"decode T={T}")


def test_matches_the_prefill_path(cuda_device):
    """The last rows of lwm_attn_fwd on the whole sequence and decode of those rows agree
    to the rounding of the two computations."""
    B, S, H, T = 1, 2048, 8, 4
    x = I.make_inputs(I.custom(B, S, H, 128, None, seed=11), cuda_device, with_dout=False)
    out_f, lse_f, _ = lwm.forward(x["q"], x["k"], x["v"])
    q = x["q"][:, S - T:].contiguous()
    out_d, lse_d, _ = lwm.decode(q, x["k"], x["v"])
    assert float((out_d.float() - out_f[:, S - T:].float()).abs().max()) <= 1e-2
    assert float((lse_d - lse_f[:, :, S - T:]).abs().max()) <= 1e-3


def test_bad_lengths_are_reported(cuda_device):
    B, S_max, H, T = 2, 512, 16, 2
    q_full, q, k, v, lens, pos = _case(B, S_max, H, T, [512, 300], cuda_device, seed=5)
    lens[1] = 1                                    # < T
    out, lse, ws = lwm.decode(q, k, v, lens)
    assert lwm.lwm_attn_check(ws) == 8
    assert torch.all(out[1] == 0) and torch.all(torch.isneginf(lse[1]))
    ref_o, ref_l = _reference(q_full[:1], k[:1], v[:1], pos[:1])
    assert_fwd(f64(out[:1]), f64(lse[:1]), ref_o, ref_l, "good row next to a bad one")
    lens[1] = S_max + 1                            # > S_max
    lwm.lwm_attn_decode(q, k, v, lens, out, lse, ws)
    assert lwm.lwm_attn_check(ws) == 8
    assert lwm.lwm_attn_check(ws) == 0


@pytest.mark.parametrize("T", [1, 4])
def test_one_million_token_cache(cuda_device, T):
    """One row, a 2^20-token cache, 32 heads: four heads against the oracle (each query
    row is exact from the row alone)."""
    B, S, H = 1, 1 << 20, 32
    g = torch.Generator(device=cuda_device)
    g.manual_seed(T)
    k = torch.randn((B, S, H, 128), generator=g, device=cuda_device, dtype=torch.bfloat16)
    v = torch.randn((B, S, H, 128), generator=g, device=cuda_device, dtype=torch.bfloat16)
    q = torch.randn((B, T, H, 128), generator=g, device=cuda_device, dtype=torch.bfloat16)
    out, lse, ws = lwm.decode(q, k, v)
    assert lwm.lwm_attn_check(ws) == 0
    heads = (0, 9, 18, 31)
    got_o, got_l, ref_o, ref_l = [], [], [], []
    for h in heads:
        kh, vh = (f64(t[:, :, h:h + 1]) for t in (k, v))
        qh = np.zeros((1, S, 1, 128))
        qh[0, S - T:, 0] = f64(q[0, :, h])
        o, l = oracle.attention_forward_rows(qh, kh, vh, None, 0, np.arange(S - T, S))
        ref_o.append(o[:, 0]); ref_l.append(l[0])
        got_o.append(f64(out[0, :, h])); got_l.append(f64(lse[0, h]))
    assert_fwd(np.stack(got_o), np.stack(got_l), np.stack(ref_o), np.stack(ref_l), f"1M cache T={T}")
