"""The public API under the double-buffered pattern a caller streaming batches uses (and
the bench's end-to-end leg times): step i's inputs upload on one copy stream while step
i - 1 computes on a compute stream, and its results download on another copy stream
while step i + 1 computes. Every step's downloaded results must equal, bit for bit, those
of the same step run alone on the default stream (the kernels are deterministic), and the
steps must not see each other's data.
"""

import pytest
import torch

import blockwise_ringattention_causal_b300 as lwm
from blockwise_ringattention_causal_b300 import inputs as I

pytestmark = pytest.mark.gpu

NAMES = ("out", "lse", "dq", "dk", "dv")


def _step_alone(x, ws):
    out, lse, _ = lwm.forward(x["q"], x["k"], x["v"], x["seg"], x["pos"], workspace=ws)
    dq, dk, dv = lwm.backward(x["q"], x["k"], x["v"], out, x["dout"], lse, x["seg"], x["pos"], workspace=ws)
    torch.cuda.synchronize()
    assert lwm.lwm_attn_check(ws) == 0
    return [t.cpu() for t in (out, lse, dq, dk, dv)]


def test_double_buffered_steps_match_steps_run_alone(cuda_device):
    # three batches of one packed shape (different seeds, same document lengths)
    steps = [I.custom(2, 1500, 4, 128, [[700, 800], [300, 1000, 200]], seed=s) for s in (11, 12, 13)]
    hosts = []
    for w in steps:
        x = I.make_inputs(w, "cpu")
        hosts.append({n: t.pin_memory() for n, t in x.items() if t is not None})
    w0 = steps[0]
    ws = lwm.new_workspace(w0.B, w0.S, w0.H, w0.D, cuda_device)

    expected = [_step_alone({n: t.to(cuda_device) for n, t in h.items()}, ws) for h in hosts]

    comp, up, down = (torch.cuda.Stream(cuda_device) for _ in range(3))
    dev_in = [{n: torch.empty_like(t, device=cuda_device) for n, t in hosts[0].items()} for _ in range(2)]
    got = [{n: None for n in NAMES} for _ in steps]
    in_free = [None, None]
    for i, h in enumerate(hosts):
        bi = i % 2
        if in_free[bi] is not None:
            up.wait_event(in_free[bi])
        with torch.cuda.stream(up):
            for n, t in h.items():
                dev_in[bi][n].copy_(t, non_blocking=True)
        ready = torch.cuda.Event()
        ready.record(up)
        comp.wait_event(ready)
        d = dev_in[bi]
        with torch.cuda.stream(comp):
            out, lse, _ = lwm.forward(d["q"], d["k"], d["v"], d["seg"], d["pos"], workspace=ws, stream=comp)
            fwd_done = torch.cuda.Event()
            fwd_done.record(comp)
            dq, dk, dv = lwm.backward(d["q"], d["k"], d["v"], out, d["dout"], lse, d["seg"], d["pos"],
                                      workspace=ws, stream=comp)
            done = torch.cuda.Event()
            done.record(comp)
        in_free[bi] = done
        down.wait_event(fwd_done)
        with torch.cuda.stream(down):
            for n, t in (("out", out), ("lse", lse)):
                got[i][n] = torch.empty(t.shape, dtype=t.dtype).pin_memory()
                got[i][n].copy_(t, non_blocking=True)
        down.wait_event(done)
        with torch.cuda.stream(down):
            for n, t in (("dq", dq), ("dk", dk), ("dv", dv)):
                got[i][n] = torch.empty(t.shape, dtype=t.dtype).pin_memory()
                got[i][n].copy_(t, non_blocking=True)
        for t in (out, lse, dq, dk, dv):
            t.record_stream(down)
    torch.cuda.synchronize()
    assert lwm.lwm_attn_check(ws) == 0

    for i in range(len(steps)):
        for k, n in enumerate(NAMES):
            assert torch.equal(got[i][n], expected[i][k]), (i, n)
    # the batches differ, so equal results across steps would mean a stale buffer
    assert not torch.equal(expected[0][2], expected[1][2])
