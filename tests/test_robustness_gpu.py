"""Failure detection and scheduling robustness on the GPU.

  * A bounded pipeline wait that runs out: a test-only short bound makes the kernels'
    waits give up; the call must report LWM_ERR_TIMEOUT through lwm_attn_check, and the
    same CUDA context and workspace must then compute correct results with the default
    bound (the kernels let in-flight copies and products land, free their tensor
    memory and return). No fault, trap or hang is involved: every wait is bounded.
  * The longest-first work list keeps its order when costs exceed the sort's bins
    (S = 1M: a forward query-tile pair costs up to 16384 key tiles).
  * A second CUDA device, when there is one, gets its own kernel attributes.
"""

import numpy as np
import pytest
import torch

import blockwise_ringattention_causal_b300 as lwm
from blockwise_ringattention_causal_b300 import inputs as I
import oracle
from tests._parity import GRAD_REL, assert_fwd, f64, rel_l2

pytestmark = pytest.mark.gpu

TIMEOUT = 7


def _fwd_bwd(x, ws):
    B, S, H, D = x["q"].shape
    out = torch.empty_like(x["q"])
    lse = torch.empty((B, H, S), dtype=torch.float32, device=x["q"].device)
    lwm.lwm_attn_fwd(x["q"], x["k"], x["v"], x["seg"], x["pos"], out, lse, ws)
    st_fwd = lwm.lwm_attn_check(ws)
    dq, dk, dv = (torch.empty_like(x["q"]) for _ in range(3))
    lwm.lwm_attn_bwd(x["q"], x["k"], x["v"], out, x["dout"], lse, x["seg"], x["pos"], dq, dk, dv, ws)
    st_bwd = lwm.lwm_attn_check(ws)
    return st_fwd, st_bwd, (out, lse, dq, dk, dv)


@pytest.fixture
def short_wait_bound():
    """Sets the process-wide wait bound to 1 ns (a wait not satisfied at once gives up) and
    restores the default afterwards, whatever the test's outcome."""
    lwm.lwm_attn_set_wait_limit(1)
    try:
        yield
    finally:
        lwm.lwm_attn_set_wait_limit(0)


def test_expired_wait_is_reported_and_the_context_stays_usable(cuda_device, short_wait_bound):
    w = I.workload(1)                     # packed 300/424/300, S = 1K, H = 4
    x = I.make_inputs(w, cuda_device)
    ws = lwm.new_workspace(w.B, w.S, w.H, w.D, cuda_device)
    st_fwd, st_bwd, _ = _fwd_bwd(x, ws)
    assert st_fwd == TIMEOUT and st_bwd == TIMEOUT, (st_fwd, st_bwd)
    # the fused backward kernel takes the same path
    out = torch.empty_like(x["q"])
    lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=cuda_device)
    lwm.lwm_attn_set_wait_limit(0)
    lwm.lwm_attn_fwd(x["q"], x["k"], x["v"], x["seg"], x["pos"], out, lse, ws)
    assert lwm.lwm_attn_check(ws) == 0
    lwm.lwm_attn_set_wait_limit(1)
    dq, dk, dv = (torch.empty_like(x["q"]) for _ in range(3))
    lwm.lwm_attn_bwd_stages(x["q"], x["k"], x["v"], out, x["dout"], lse, dq, dk, dv,
                            lwm.LWM_BWD_DELTA | lwm.LWM_BWD_FUSED, ws)
    assert lwm.lwm_attn_check(ws) == TIMEOUT

    # default bound again: same context, same workspace, correct results
    lwm.lwm_attn_set_wait_limit(0)
    st_fwd, st_bwd, (out, lse, dq, dk, dv) = _fwd_bwd(x, ws)
    assert st_fwd == 0 and st_bwd == 0
    seg = x["seg"].cpu().numpy()
    ref_o, ref_l = oracle.attention_forward(f64(x["q"]), f64(x["k"]), f64(x["v"]), seg)
    assert_fwd(f64(out), f64(lse), ref_o, ref_l, "after an expired wait")
    refs = oracle.attention_backward(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["dout"]), seg)
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        assert rel_l2(f64(g), r) <= GRAD_REL, name


def _align256(n):
    return (n + 255) & ~255


def test_longest_first_order_at_1m_tokens(cuda_device):
    """One causal document of 2^20 tokens: query-tile pair p costs (2p + 1) + (2p + 2) key
    tiles, all distinct at the sort's granularity, so the forward list must be exactly
    the pairs in descending order."""
    B, S, H, D = 1, 1 << 20, 32, 128
    ws = lwm.new_workspace(B, S, H, D, cuda_device, forward_only=True)
    lwm.lwm_attn_prepare(None, None, B, S, H, D, 1, ws)
    assert lwm.lwm_attn_check(ws) == 0
    nT = S // 128
    nP = nT // 2
    # workspace layout: 256-byte header, lo [B, nT * 128], kend [B, nT], forward list [B, nP]
    off_list = 256 + _align256(B * S * 4) + _align256(B * nT * 4)
    lst = ws[off_list:off_list + 4 * nP].view(torch.int32).cpu().numpy()
    np.testing.assert_array_equal(lst, np.arange(nP - 1, -1, -1))


def test_second_device_gets_its_own_kernel_attributes():
    if torch.cuda.device_count() < 2:
        pytest.skip("one CUDA device")
    w = I.custom(1, 700, 2, 128, [[300, 400]], seed=3)
    for d in (0, 1):
        dev = torch.device("cuda", d)
        with torch.cuda.device(dev):
            x = I.make_inputs(w, dev)
            out, lse, ws = lwm.forward(x["q"], x["k"], x["v"], x["seg"], x["pos"])
            dq, dk, dv = lwm.backward(x["q"], x["k"], x["v"], out, x["dout"], lse, x["seg"], x["pos"], ws)
            assert lwm.lwm_attn_check(ws) == 0
            seg = x["seg"].cpu().numpy()
            ref_o, ref_l = oracle.attention_forward(f64(x["q"]), f64(x["k"]), f64(x["v"]), seg)
            assert_fwd(f64(out), f64(lse), ref_o, ref_l, f"device {d}")
