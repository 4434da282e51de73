"""Exact causal, segment-masked (packed) softmax attention for B300 (sm_103a).

A thin ctypes binding over the C ABI of ``liblwm_attn.so`` (declared in
``include/lwm_attn.h``): the functions below only check and marshal torch tensors
into pointers and sizes; every step of the computation runs in the library's CUDA
kernels. There is no CPU fallback: without the built library every call raises.

Attention computed (LWM, "World Model on Million-Length Video And Language With
Blockwise RingAttention"; deep-dive page, sections "RingAttention 为什么必要",
"模型结构" and "Masked sequence packing"): exact softmax(q k^T / sqrt(D)) v, causal,
with several documents packed in one row attending only to themselves.
"""

from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "LwmError", "library_path", "load_library",
    "lwm_attn_workspace_size", "lwm_attn_workspace_size_fwd", "lwm_attn_prepare", "lwm_attn_fwd", "lwm_attn_fwd_ring",
    "lwm_attn_fwd_prepared", "lwm_attn_bwd", "lwm_attn_bwd_prepared", "lwm_attn_bwd_stages",
    "lwm_attn_check", "lwm_attn_set_wait_limit", "lwm_attn_rope", "rope",
    "lwm_attn_decode_workspace_size", "lwm_attn_decode", "decode",
    "lwm_packed_loss_workspace_size", "lwm_packed_loss", "packed_loss",
    "lwm_status_string", "lwm_last_error", "new_workspace", "forward", "backward",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None

STATUS_NAMES = {
    0: "LWM_OK", 1: "LWM_ERR_INVALID_ARG", 2: "LWM_ERR_UNSUPPORTED", 3: "LWM_ERR_ALIGNMENT",
    4: "LWM_ERR_SEGMENTS", 5: "LWM_ERR_WORKSPACE", 6: "LWM_ERR_CUDA", 7: "LWM_ERR_TIMEOUT",
    8: "LWM_ERR_LENGTHS", 9: "LWM_ERR_TARGETS",
}

# name -> (restype, argtypes)
_P, _I, _Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
_SIGNATURES = {
    "lwm_attn_workspace_size": (_Z, [_I, _I, _I, _I]),
    "lwm_attn_workspace_size_fwd": (_Z, [_I, _I, _I, _I]),
    "lwm_attn_prepare": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _Z, _P]),
    "lwm_attn_fwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _Z, _P]),
    "lwm_attn_fwd_ring": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _Z, _P]),
    "lwm_attn_fwd_prepared": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _Z, _P]),
    "lwm_attn_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _Z, _P]),
    "lwm_attn_bwd_prepared": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _Z, _P]),
    "lwm_attn_bwd_stages": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, ctypes.c_uint, _P, _Z, _P]),
    "lwm_attn_check": (_I, [_P, _P]),
    "lwm_status_string": (ctypes.c_char_p, [_I]),
    "lwm_last_error": (ctypes.c_char_p, []),
    "lwm_attn_fwd_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P]),
    "lwm_attn_set_wait_limit": (_I, [ctypes.c_uint64]),
    "lwm_attn_rope": (_I, [_P, _P, _P, ctypes.c_double, _P, _P, _I, _I, _I, _I, _I, _P]),
    "lwm_attn_decode_workspace_size": (_Z, [_I, _I, _I, _I, _I]),
    "lwm_attn_decode": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _Z, _P]),
    "lwm_packed_loss_workspace_size": (_Z, [_I, _I]),
    "lwm_packed_loss": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _Z, _P]),
}


class LwmError(RuntimeError):
    """A non-zero lwm_status returned by the library."""

    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {lwm_status_string(status)}")


def library_path() -> str:
    return os.path.join(_HERE, "liblwm_attn.so")


def load_library():
    """Load liblwm_attn.so (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -m blockwise_ringattention_causal_b300.build`")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


def lwm_status_string(status: int) -> str:
    try:
        return load_library().lwm_status_string(int(status)).decode()
    except RuntimeError:
        return STATUS_NAMES.get(int(status), f"status {status}")


def lwm_last_error() -> str:
    return load_library().lwm_last_error().decode()


def _check(status: int, where: str):
    if status != 0:
        if status == 6:
            where = f"{where} [{lwm_last_error()}]"
        raise LwmError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _shape(q):
    if q.dim() != 4:
        raise ValueError("expected a [B, S, H, D] tensor")
    return tuple(int(x) for x in q.shape)


def _need(t, name, dtype, shape=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _seg(seg, pos, B, S):
    for t, n in ((seg, "seg_ids"), (pos, "pos")):
        if t is not None:
            _need(t, n, torch.int32, (B, S))


def lwm_attn_workspace_size(B, S, H, D) -> int:
    return int(load_library().lwm_attn_workspace_size(B, S, H, D))


def lwm_attn_workspace_size_fwd(B, S, H, D) -> int:
    return int(load_library().lwm_attn_workspace_size_fwd(B, S, H, D))


def new_workspace(B, S, H, D, device="cuda", forward_only=False) -> torch.Tensor:
    """A zero-filled workspace (the library requires zeros before first use).
    ``forward_only`` leaves out the dQ accumulator that only the backward pass uses."""
    n = (lwm_attn_workspace_size_fwd if forward_only else lwm_attn_workspace_size)(B, S, H, D)
    if n == 0:
        raise ValueError("unsupported sizes")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def lwm_attn_prepare(seg_ids, pos, B, S, H, D, kv_chunks, workspace, stream=None):
    _seg(seg_ids, pos, B, S)
    _check(load_library().lwm_attn_prepare(_ptr(seg_ids), _ptr(pos), B, S, H, D, kv_chunks,
                                           _ptr(workspace), workspace.numel(), _stream(stream)),
           "lwm_attn_prepare")


def lwm_attn_fwd(q, k, v, seg_ids, pos, out, lse, workspace, stream=None):
    B, S, H, D = _shape(q)
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out")):
        _need(t, n, torch.bfloat16, (B, S, H, D))
    _need(lse, "lse", torch.float32, (B, H, S))
    _seg(seg_ids, pos, B, S)
    _check(load_library().lwm_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(seg_ids), _ptr(pos), _ptr(out),
                                       _ptr(lse), B, S, H, D, _ptr(workspace), workspace.numel(),
                                       _stream(stream)), "lwm_attn_fwd")


def lwm_attn_fwd_ring(q, k, v, seg_ids, pos, out, lse, kv_chunks, workspace, stream=None):
    B, S, H, D = _shape(q)
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out")):
        _need(t, n, torch.bfloat16, (B, S, H, D))
    _need(lse, "lse", torch.float32, (B, H, S))
    _seg(seg_ids, pos, B, S)
    _check(load_library().lwm_attn_fwd_ring(_ptr(q), _ptr(k), _ptr(v), _ptr(seg_ids), _ptr(pos), _ptr(out),
                                            _ptr(lse), B, S, H, D, int(kv_chunks), _ptr(workspace),
                                            workspace.numel(), _stream(stream)), "lwm_attn_fwd_ring")


def lwm_attn_fwd_prepared(q, k, v, out, lse, workspace, stream=None):
    B, S, H, D = _shape(q)
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out")):
        _need(t, n, torch.bfloat16, (B, S, H, D))
    _need(lse, "lse", torch.float32, (B, H, S))
    _check(load_library().lwm_attn_fwd_prepared(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, S, H, D,
                                                _ptr(workspace), workspace.numel(), _stream(stream)),
           "lwm_attn_fwd_prepared")


def lwm_attn_bwd(q, k, v, out, dout, lse, seg_ids, pos, dq, dk, dv, workspace, stream=None):
    B, S, H, D = _shape(q)
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout"), (dq, "dq"), (dk, "dk"),
                 (dv, "dv")):
        _need(t, n, torch.bfloat16, (B, S, H, D))
    _need(lse, "lse", torch.float32, (B, H, S))
    _seg(seg_ids, pos, B, S)
    _check(load_library().lwm_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse),
                                       _ptr(seg_ids), _ptr(pos), _ptr(dq), _ptr(dk), _ptr(dv), B, S, H, D,
                                       _ptr(workspace), workspace.numel(), _stream(stream)), "lwm_attn_bwd")


def lwm_attn_bwd_prepared(q, k, v, out, dout, lse, dq, dk, dv, workspace, stream=None):
    B, S, H, D = _shape(q)
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout"), (dq, "dq"), (dk, "dk"),
                 (dv, "dv")):
        _need(t, n, torch.bfloat16, (B, S, H, D))
    _need(lse, "lse", torch.float32, (B, H, S))
    _check(load_library().lwm_attn_bwd_prepared(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse),
                                                _ptr(dq), _ptr(dk), _ptr(dv), B, S, H, D, _ptr(workspace),
                                                workspace.numel(), _stream(stream)), "lwm_attn_bwd_prepared")


LWM_BWD_DELTA, LWM_BWD_DKDV, LWM_BWD_DQ, LWM_BWD_ALL, LWM_BWD_FUSED = 1, 2, 4, 7, 8


def lwm_attn_bwd_stages(q, k, v, out, dout, lse, dq, dk, dv, stages, workspace, stream=None):
    """Selected backward stages (bit mask of LWM_BWD_*); unused tensors may be None."""
    B, S, H, D = _shape(q if q is not None else out)
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout"), (dq, "dq"), (dk, "dk"),
                 (dv, "dv")):
        if t is not None:
            _need(t, n, torch.bfloat16, (B, S, H, D))
    if lse is not None:
        _need(lse, "lse", torch.float32, (B, H, S))
    _check(load_library().lwm_attn_bwd_stages(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse),
                                              _ptr(dq), _ptr(dk), _ptr(dv), B, S, H, D, int(stages),
                                              _ptr(workspace), workspace.numel(), _stream(stream)),
           "lwm_attn_bwd_stages")


def lwm_attn_rope(q, k, pos, theta, q_out, k_out, inverse=False, stream=None):
    """RoPE rotation (or, with ``inverse``, its transpose) of q and/or k by ``pos``.

    Either of (q, q_out) and (k, k_out) may be (None, None); out may be the input."""
    ref = q if q is not None else k
    B, S, H, D = _shape(ref)
    for t, n in ((q, "q"), (k, "k"), (q_out, "q_out"), (k_out, "k_out")):
        if t is not None:
            _need(t, n, torch.bfloat16, (B, S, H, D))
    if pos is not None:
        _need(pos, "pos", torch.int32, (B, S))
    _check(load_library().lwm_attn_rope(_ptr(q), _ptr(k), _ptr(pos), float(theta), _ptr(q_out), _ptr(k_out),
                                        B, S, H, D, int(bool(inverse)), _stream(stream)), "lwm_attn_rope")


def rope(q, k, pos, theta, inverse=False, stream=None):
    """Rotated copies (q_rot, k_rot) of q and k (either may be None)."""
    q_out = None if q is None else torch.empty_like(q)
    k_out = None if k is None else torch.empty_like(k)
    lwm_attn_rope(q, k, pos, theta, q_out, k_out, inverse, stream)
    return q_out, k_out


def lwm_attn_decode_workspace_size(B, T, S_max, H, D) -> int:
    return int(load_library().lwm_attn_decode_workspace_size(B, T, S_max, H, D))


def lwm_attn_decode(q, k_cache, v_cache, kv_len, out, lse, workspace, stream=None):
    """Attention of the T newest tokens (q [B, T, H, D]) against the caches [B, S_max, H, D]."""
    B, T, H, D = _shape(q)
    S_max = int(k_cache.shape[1])
    _need(q, "q", torch.bfloat16)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, torch.bfloat16, (B, S_max, H, D))
    _need(out, "out", torch.bfloat16, (B, T, H, D))
    _need(lse, "lse", torch.float32, (B, H, T))
    if kv_len is not None:
        _need(kv_len, "kv_len", torch.int32, (B,))
    _check(load_library().lwm_attn_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kv_len), _ptr(out), _ptr(lse),
                                          B, T, S_max, H, D, _ptr(workspace), workspace.numel(), _stream(stream)),
           "lwm_attn_decode")


def decode(q, k_cache, v_cache, kv_len=None, workspace=None, stream=None):
    """Allocate out/lse (and a workspace if none is given) and decode. Returns (out, lse, workspace)."""
    B, T, H, D = _shape(q)
    out = torch.empty_like(q)
    lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    if workspace is None:
        n = lwm_attn_decode_workspace_size(B, T, int(k_cache.shape[1]), H, D)
        if n == 0:
            raise ValueError("unsupported decode sizes")
        workspace = torch.zeros(n, dtype=torch.uint8, device=q.device)
    lwm_attn_decode(q, k_cache, v_cache, kv_len, out, lse, workspace, stream)
    return out, lse, workspace


def lwm_packed_loss_workspace_size(B, S) -> int:
    return int(load_library().lwm_packed_loss_workspace_size(B, S))


def lwm_packed_loss(logits, targets, weight, seg_ids, loss, dlogits, workspace, stream=None):
    """Re-weighted packed cross-entropy: loss (float64 [1]) and, if given, dlogits."""
    if logits.dim() != 3:
        raise ValueError("logits must be [B, S, V]")
    B, S, V = (int(x) for x in logits.shape)
    _need(logits, "logits", torch.bfloat16)
    _need(targets, "targets", torch.int32, (B, S))
    if weight is not None:
        _need(weight, "weight", torch.float32, (B, S))
    if seg_ids is not None:
        _need(seg_ids, "seg_ids", torch.int32, (B, S))
    _need(loss, "loss", torch.float64)
    if dlogits is not None:
        _need(dlogits, "dlogits", torch.bfloat16, (B, S, V))
    _check(load_library().lwm_packed_loss(_ptr(logits), _ptr(targets), _ptr(weight), _ptr(seg_ids), _ptr(loss),
                                          _ptr(dlogits), B, S, V, _ptr(workspace), workspace.numel(),
                                          _stream(stream)), "lwm_packed_loss")


def packed_loss(logits, targets, weight=None, seg_ids=None, grad=True, workspace=None, stream=None):
    """Allocate the outputs and run lwm_packed_loss. Returns (loss [1] float64, dlogits or None, workspace)."""
    B, S, V = (int(x) for x in logits.shape)
    loss = torch.empty(1, dtype=torch.float64, device=logits.device)
    dlogits = torch.empty_like(logits) if grad else None
    if workspace is None:
        workspace = torch.zeros(lwm_packed_loss_workspace_size(B, S), dtype=torch.uint8, device=logits.device)
    lwm_packed_loss(logits, targets, weight, seg_ids, loss, dlogits, workspace, stream)
    return loss, dlogits, workspace


def lwm_attn_set_wait_limit(limit_ns):
    """Bound of the kernels' pipeline waits for every later launch of this process (0 = 2 s)."""
    _check(load_library().lwm_attn_set_wait_limit(int(limit_ns)), "lwm_attn_set_wait_limit")


def lwm_attn_check(workspace, stream=None) -> int:
    """Synchronise and return (and clear) the device error status; 0 = LWM_OK."""
    return int(load_library().lwm_attn_check(_ptr(workspace), _stream(stream)))


def forward(q, k, v, seg_ids=None, pos=None, kv_chunks=1, workspace=None, stream=None):
    """Allocate out/lse and run the forward pass. Returns (out, lse, workspace)."""
    B, S, H, D = _shape(q)
    out = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = new_workspace(B, S, H, D, q.device)
    if kv_chunks == 1:
        lwm_attn_fwd(q, k, v, seg_ids, pos, out, lse, workspace, stream)
    else:
        lwm_attn_fwd_ring(q, k, v, seg_ids, pos, out, lse, kv_chunks, workspace, stream)
    return out, lse, workspace


def backward(q, k, v, out, dout, lse, seg_ids=None, pos=None, workspace=None, stream=None, fused=False):
    """Allocate dq/dk/dv and run the backward pass. Returns (dq, dk, dv).

    The default runs lwm_attn_bwd (row-dot pre-pass, dK/dV kernel, dQ kernel; every
    gradient bitwise reproducible). ``fused=True`` runs the metadata pre-pass and the
    LWM_BWD_DELTA | LWM_BWD_FUSED stages (one dK/dV/dQ kernel, dq summed in fp32 in a
    scheduling-dependent order)."""
    B, S, H, D = _shape(q)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if workspace is None:
        workspace = new_workspace(B, S, H, D, q.device)
    if fused:
        lwm_attn_prepare(seg_ids, pos, B, S, H, D, 1, workspace, stream)
        lwm_attn_bwd_stages(q, k, v, out, dout, lse, dq, dk, dv, LWM_BWD_DELTA | LWM_BWD_FUSED, workspace, stream)
    else:
        lwm_attn_bwd(q, k, v, out, dout, lse, seg_ids, pos, dq, dk, dv, workspace, stream)
    return dq, dk, dv
