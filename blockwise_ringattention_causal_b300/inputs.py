"""Seeded synthetic inputs for the attention workloads (no attention arithmetic here).

The workloads stand in for the data the LWM pages train on (text documents, images
and videos tokenised at 256 VQGAN codes per frame, packed into long rows; LWM
deep-dive page, sections "模型结构", "Masked sequence packing" and the data-mix
table). Those datasets are not used: only their shapes, lengths and packing
structure are reproduced, with Gaussian values.

Conventions:
  * q, k, v, dout: bf16 [B, S, H, D], drawn N(0, 1) in float32 from one
    ``torch.Generator`` seeded with ``seed`` on ``device`` (in the order q, k, v,
    dout, then any per-frame offsets), then rounded to bf16;
  * seg: int32 [B, S] document id per token, 0, 1, 2, ... per row, contiguous runs;
    pos: int32 [B, S] position within the document, restarting at 0.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

TEXT_MIN, TEXT_MAX = 1024, 16384
IMAGE_DOC = 258          # <vision> + 256 VQGAN codes + <eof>
FRAME_TOKENS = 256       # VQGAN tokens per frame


@dataclass
class Workload:
    """One named attention workload: shapes plus the document lengths of each row."""

    name: str
    B: int
    S: int
    H: int
    D: int
    lengths: list = field(default_factory=list)   # per row: list of document lengths
    backward: bool = True
    frame_offset_std: float = 0.0                 # per-frame mean offset (video)
    kv_chunks: int = 1                            # ring-ordered KV chunks in one launch
    seed: int = 0

    def describe(self):
        return {"workload": self.name, "B": self.B, "S": self.S, "H": self.H, "D": self.D,
                "docs_per_row": [len(r) for r in self.lengths],
                "kv_chunks": self.kv_chunks, "backward": self.backward, "seed": self.seed}


def packed_mixed_lengths(S, rows, seed=0):
    """Document lengths for rows packed with alternating text and image documents.

    One ``numpy.random.default_rng(seed)`` stream is shared by all rows. Each row
    starts with a text document; text lengths are round(exp(U(ln 1024, ln 16384)))
    (log-uniform in [1K, 16K]); image documents are 258 tokens; the last document of
    a row is cut so that the row is exactly ``S`` tokens.
    """
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(rows):
        lens, filled, text = [], 0, True
        while filled < S:
            if text:
                L = int(round(math.exp(rng.uniform(math.log(TEXT_MIN), math.log(TEXT_MAX)))))
            else:
                L = IMAGE_DOC
            L = min(L, S - filled)
            lens.append(L)
            filled += L
            text = not text
        out.append(lens)
    return out


def workload(config: int, seed: int = 0) -> Workload:
    """The five named workloads (1: packed 1K, 2: 32K causal, 3: 64K mixed packing,
    4: 256K video, 5: 1M forward in 8 ring-ordered KV chunks)."""
    if config == 1:
        return Workload("packed-3doc-S1K-H4", 1, 1024, 4, 128, [[300, 424, 300]], seed=seed)
    if config == 2:
        return Workload("causal-S32K-H32-D128", 1, 32768, 32, 128, [[32768]], seed=seed)
    if config == 3:
        S = 65536
        return Workload("packed-mixed-S64K-B2-H32", 2, S, 32, 128, packed_mixed_lengths(S, 2, seed), seed=seed)
    if config == 4:
        S = 1024 * FRAME_TOKENS
        return Workload("video-S256K-H32", 1, S, 32, 128, [[S]], frame_offset_std=0.5, seed=seed)
    if config == 5:
        S = 1 << 20
        return Workload("causal-S1M-H32-fwd", 1, S, 32, 128, [[S]], backward=False, kv_chunks=8, seed=seed)
    raise ValueError(f"unknown workload {config}")


def custom(B, S, H, D, lengths=None, seed=0, backward=True, kv_chunks=1, frame_offset_std=0.0, name="custom"):
    """An arbitrary workload; ``lengths`` defaults to one document per row.

    A row whose lengths sum to less than S is padded with a trailing run of
    seg = -1 tokens (pos = 0 there).
    """
    if lengths is None:
        lengths = [[S] for _ in range(B)]
    return Workload(name, B, S, H, D, [list(map(int, r)) for r in lengths], backward,
                    frame_offset_std, kv_chunks, seed)


def segments(w: Workload):
    """(seg, pos) int32 numpy arrays [B, S] for the workload's document lengths."""
    seg = np.full((w.B, w.S), -1, np.int32)
    pos = np.zeros((w.B, w.S), np.int32)
    for b, lens in enumerate(w.lengths):
        o = 0
        for d, L in enumerate(lens):
            seg[b, o:o + L] = d
            pos[b, o:o + L] = np.arange(L, dtype=np.int32)
            o += L
        if o > w.S:
            raise ValueError("document lengths exceed S")
    return seg, pos


def pairs_per_head(w: Workload) -> int:
    """Visible (query, key) pairs per head from the document lengths: sum L(L+1)/2."""
    return int(sum(L * (L + 1) // 2 for lens in w.lengths for L in lens))


def make_inputs(w: Workload, device="cpu", with_dout=True):
    """Tensors for the workload: dict with q, k, v, (dout), seg, pos on ``device``."""
    g = torch.Generator(device=device)
    g.manual_seed(w.seed)
    shape = (w.B, w.S, w.H, w.D)

    def draw():
        return torch.randn(shape, generator=g, device=device, dtype=torch.float32)

    q, k, v = draw(), draw(), draw()
    dout = draw() if with_dout else None
    if w.frame_offset_std > 0.0:
        frames = w.S // FRAME_TOKENS
        for t in (q, k, v):
            off = torch.randn((w.B, frames, 1, w.H, w.D), generator=g, device=device,
                              dtype=torch.float32) * w.frame_offset_std
            t.view(w.B, frames, FRAME_TOKENS, w.H, w.D).add_(off)
    seg, pos = segments(w)
    out = {"q": q.to(torch.bfloat16), "k": k.to(torch.bfloat16), "v": v.to(torch.bfloat16),
           "seg": torch.from_numpy(seg).to(device), "pos": torch.from_numpy(pos).to(device)}
    if dout is not None:
        out["dout"] = dout.to(torch.bfloat16)
    return out


def sample_rows(S, n=512, seed=1):
    """Sorted distinct query rows for sampled checks: 0, S-1 and one per stratum."""
    rng = np.random.default_rng(seed)
    if S <= n:
        return np.arange(S)
    strata = n - 2
    edges = np.linspace(1, S - 1, strata + 1).astype(np.int64)
    rows = [0, S - 1]
    for a, b in zip(edges[:-1], edges[1:]):
        rows.append(int(rng.integers(a, max(a + 1, b))))
    return np.unique(np.asarray(rows, np.int64))
