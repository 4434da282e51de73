"""Plain float64 oracle of rotary position embedding (RoPE) on q and k.

Test infrastructure only: the product path never imports this module.

What the pages fix: LWM extends LLaMA-2's context by raising RoPE's base theta as the
context grows (deep-dive page, section "Stage I：长上下文语言模型", and Tables 11
and 13: theta = 1M at 32K tokens, 10M at 128K-256K, 25M at 512K, 50M at 1M and in
every vision-language stage). The pages name RoPE but print no formula; the rotation
below is RoPE's published definition (the LLaMA lineage rotates adjacent pairs):

    for token i at position p = pos[b, i] and pair m = 0 .. D/2 - 1,
    angle      = p * theta^(-2m/D)
    y[2m]      = x[2m] cos(angle) - x[2m+1] sin(angle)
    y[2m+1]    = x[2m] sin(angle) + x[2m+1] cos(angle)

and the inverse (the transpose, used for gradients) rotates by -angle. Attention with
RoPE is the attention oracle applied to the rotated q and k (v unrotated); its
gradients with respect to the unrotated q and k are the inverse rotations of the
gradients with respect to the rotated ones.

Storage reading: the rotated q and k are the attention's inputs, whose type is bf16,
so :func:`attention_forward_rope` rounds the float64 rotation to bf16 (round to
nearest, ties to even) before the attention, as a kernel that writes rotated bf16
tensors does. The gradient treats that rounding as the identity (it is storage).
"""

from __future__ import annotations

import numpy as np

from .attention import attention_backward, attention_forward


def rope_angles(pos, theta, D):
    """angle[b, i, m] = pos[b, i] * theta^(-2m/D), float64 [B, S, D/2]."""
    m = np.arange(D // 2, dtype=np.float64)
    inv_freq = np.power(float(theta), -2.0 * m / D)
    return np.asarray(pos, dtype=np.float64)[..., None] * inv_freq


def rope_rotate(x, pos, theta, inverse=False):
    """Rotate the adjacent pairs (2m, 2m+1) of x [B, S, H, D] by pos * theta^(-2m/D)
    (by the negative angle when ``inverse``). float64."""
    x = np.asarray(x, dtype=np.float64)
    B, S, H, D = x.shape
    ang = rope_angles(pos, theta, D)
    if inverse:
        ang = -ang
    c = np.cos(ang)[:, :, None, :]
    s = np.sin(ang)[:, :, None, :]
    x0, x1 = x[..., 0::2], x[..., 1::2]
    y = np.empty_like(x)
    y[..., 0::2] = x0 * c - x1 * s
    y[..., 1::2] = x0 * s + x1 * c
    return y


def round_bf16(x):
    """Round float64 values to the nearest bfloat16 value (8 significant bits, ties to
    even), returned as float64. Magnitudes stay in the normal range here."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                      # x = m * 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)


def attention_forward_rope(q, k, v, seg, pos, theta, bf16_inputs=True):
    """(out, lse) of attention on RoPE-rotated q and k."""
    qr, kr = rope_rotate(q, pos, theta), rope_rotate(k, pos, theta)
    if bf16_inputs:
        qr, kr = round_bf16(qr), round_bf16(kr)
    return attention_forward(qr, kr, v, seg)


def attention_backward_rope(q, k, v, dout, seg, pos, theta, bf16_inputs=True):
    """(dq, dk, dv) with respect to the unrotated q, k and v."""
    qr, kr = rope_rotate(q, pos, theta), rope_rotate(k, pos, theta)
    if bf16_inputs:
        qr, kr = round_bf16(qr), round_bf16(kr)
    gq, gk, gv = attention_backward(qr, kr, v, dout, seg)
    return rope_rotate(gq, pos, theta, inverse=True), rope_rotate(gk, pos, theta, inverse=True), gv
