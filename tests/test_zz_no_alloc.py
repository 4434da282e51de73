"""lwm_attn_fwd_noalloc: the forward pass for callers that cannot allocate device memory.

Such callers (a plug-in inside a framework that owns all device memory, or a path that
must not call cudaMalloc because it may synchronise the device) get a forward pass whose
workspace is a device array owned by the library. These tests call it through the C ABI
and check it against lwm_attn_fwd, which takes a caller-provided workspace (bitwise:
the kernels are the same and deterministic), and against the float64 oracle.

This file is named so that pytest collects it last.
"""

import ctypes

import numpy as np
import pytest
import torch

import blockwise_ringattention_causal_b300 as lwm
from blockwise_ringattention_causal_b300 import build as lwm_build
from blockwise_ringattention_causal_b300 import inputs as I
import oracle
from tests._parity import assert_fwd, f64


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lwm_build.build()
    lib = lwm.load_library()
    P = ctypes.c_void_p
    # 1 x 2M tokens needs more than the 16 MiB array: refused before touching a device
    assert lib.lwm_attn_fwd_noalloc(P(4096), P(4096), P(4096), None, None, P(4096), P(4096),
                                    1, 1 << 21, 32, 128, None) == 1
    assert lib.lwm_attn_fwd_noalloc(P(4096), P(4096), P(4096), None, None, P(4096), P(4096),
                                    1, 1024, 4, 64, None) == 2


@pytest.mark.gpu
def test_noalloc_matches_workspace_forward_twice(cuda_device):
    lib = lwm.load_library()
    stream = torch.cuda.current_stream()
    sp = ctypes.c_void_p(stream.cuda_stream)
    # a packed row and a second row with padding, ragged S, several heads
    w = I.custom(2, 1000, 4, 128, [[300, 1, 450, 249], [600, 350]], seed=21)
    x = I.make_inputs(w, cuda_device, with_dout=False)
    B, S, H, D = w.B, w.S, w.H, w.D
    ref_out, ref_lse, ws = lwm.forward(x["q"], x["k"], x["v"], x["seg"], x["pos"])
    assert lwm.lwm_attn_check(ws) == 0

    results = []
    for call in range(2):
        out = torch.full_like(x["q"], float("nan"))
        lse = torch.full((B, H, S), float("nan"), dtype=torch.float32, device=cuda_device)
        st = lib.lwm_attn_fwd_noalloc(_p(x["q"]), _p(x["k"]), _p(x["v"]), _p(x["seg"]), _p(x["pos"]), _p(out),
                                      _p(lse), B, S, H, D, sp)
        assert st == 0, lwm.lwm_status_string(st)
        torch.cuda.synchronize()
        results.append((out, lse))
        # the same deterministic kernels as lwm_attn_fwd: bitwise equal results
        assert torch.equal(out, ref_out), f"no-alloc call {call + 1}: out differs from lwm_attn_fwd"
        assert torch.equal(lse, ref_lse), f"no-alloc call {call + 1}: lse differs from lwm_attn_fwd"
    # and correct: the float64 oracle at the workload tolerance
    ref_o, ref_l = oracle.attention_forward(f64(x["q"]), f64(x["k"]), f64(x["v"]), x["seg"].cpu().numpy())
    assert_fwd(f64(results[0][0]), f64(results[0][1]), ref_o, ref_l, "no-alloc against the oracle",
               bf16_bound=True)

    # a second, different problem between and after: the shared array keeps no stale state
    w2 = I.custom(1, 257, 2, 128, [[200, 57]], seed=22)
    x2 = I.make_inputs(w2, cuda_device, with_dout=False)
    out2 = torch.empty_like(x2["q"])
    lse2 = torch.empty((1, 2, 257), dtype=torch.float32, device=cuda_device)
    assert lib.lwm_attn_fwd_noalloc(_p(x2["q"]), _p(x2["k"]), _p(x2["v"]), _p(x2["seg"]), _p(x2["pos"]),
                                    _p(out2), _p(lse2), 1, 257, 2, 128, sp) == 0
    r_out2, r_lse2, ws2 = lwm.forward(x2["q"], x2["k"], x2["v"], x2["seg"], x2["pos"])
    torch.cuda.synchronize()
    assert torch.equal(out2, r_out2) and torch.equal(lse2, r_lse2), "no-alloc second problem"
    assert torch.isfinite(results[1][0].float()).all()
