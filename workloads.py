"""Seeded synthetic inputs for frame-aligned window-sparse attention.

This module holds shapes, seeds and random draws only: no attention, mask,
norm or bound arithmetic.  Both sides of a parity check (the CPU oracle and
the CUDA library) take their inputs from here and from nowhere else.

Shapes and value distributions follow the super-resolution attention the
Google Developers Blog post "HeyGen x Google Cloud: Bringing Avatar IV to
TPUs" describes in its section on deleting the mask (tens of thousands of
tokens, each frame attending a window of nearby frames plus one global
reference frame).  The pages use production activations, which are not
available; these seeded draws stand in for them:

  q ~ N(0,1), k ~ N(0,1) + a per-head offset ~ N(0, 4) shared by every token
  of the head (keys "share a large common component", section on breaking
  softmax's dependency chain), v ~ N(0,1); all cast to bf16.

Token order: the R reference frames first, then video frames 0..F-1, each
T tokens long; tensors are row-major [B, H, N, D] with N = (R + F) * T.
"""
from __future__ import annotations

import dataclasses

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    heads: int
    head_dim: int
    frames: int            # F: video frames
    ref_frames: int        # R: global reference frames (a prefix of the sequence)
    tokens_per_frame: int  # T
    window: int            # w: video frames f, g interact iff |f - g| <= w
    seed: int
    boost_heads: tuple = ()  # heads whose 1% of query rows are scaled by `boost`
    boost: float = 8.0
    description: str = ""

    @property
    def n_tokens(self) -> int:
        return (self.frames + self.ref_frames) * self.tokens_per_frame

    @property
    def scale(self) -> float:
        return 1.0 / float(self.head_dim) ** 0.5

    def label(self) -> str:
        w = "all" if self.window >= self.frames - 1 else f"+-{self.window}"
        return (f"{self.name}: B={self.batch} H={self.heads} D={self.head_dim} "
                f"F={self.frames}+{self.ref_frames}ref T={self.tokens_per_frame} "
                f"N={self.n_tokens} window={w}")


WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 64, 4, 1, 48, 1, 0,
                     description="4 frames + 1 reference, 48 tokens/frame"),
    "small": Workload("small", 1, 8, 128, 9, 1, 208, 1, 1,
                      description="9 frames + 1 reference, 13x16 tokens/frame"),
    "sr": Workload("sr", 1, 24, 128, 21, 1, 1040, 2, 2,
                   description="SR-shaped: 21 frames + 1 reference, 26x40 latent grid"),
    "sr_long": Workload("sr_long", 1, 24, 128, 25, 1, 2080, 3, 3, boost_heads=(5, 17),
                        description="SR-long: 25 frames + 1 reference; heads 5 and 17 "
                                    "have 1% of query rows scaled x8"),
    "dense": Workload("dense", 2, 40, 128, 13, 1, 1568, 12, 4,
                      description="dense-window A2V-like: 13 frames + 1 reference, 28x56, "
                                  "every frame sees every frame"),
}


def generate(wl: Workload):
    """Returns (q, k, v) as contiguous CPU bf16 tensors [B, H, N, D].

    Draw order from one torch CPU generator seeded with wl.seed:
    q, k, offset[H, D] (scaled by 2, i.e. variance 4), v; then k += offset,
    cast to bf16, then for each boosted head its rows randperm(N)[:N // 100]
    are multiplied by `boost` (exact for a power of two in bf16).
    """
    g = torch.Generator().manual_seed(wl.seed)
    shape = (wl.batch, wl.heads, wl.n_tokens, wl.head_dim)
    q = torch.randn(shape, generator=g)
    k = torch.randn(shape, generator=g)
    off = 2.0 * torch.randn((wl.heads, wl.head_dim), generator=g)
    v = torch.randn(shape, generator=g)
    k += off[None, :, None, :]
    q = q.to(torch.bfloat16)
    k = k.to(torch.bfloat16)
    v = v.to(torch.bfloat16)
    for h in wl.boost_heads:
        rows = torch.randperm(wl.n_tokens, generator=g)[: wl.n_tokens // 100]
        q[:, h, rows] = q[:, h, rows] * wl.boost
    return q.contiguous(), k.contiguous(), v.contiguous()


def sample_rows(wl: Workload, n_random: int = 256) -> list:
    """Query rows checked at full size: the first and last 16 rows of every
    frame (reference and video: the frame edges) plus n_random seeded rows."""
    T, nf, n = wl.tokens_per_frame, wl.frames + wl.ref_frames, wl.n_tokens
    rows = set()
    for f in range(nf):
        rows.update(range(f * T, min(f * T + 16, (f + 1) * T)))
        rows.update(range(max((f + 1) * T - 16, f * T), (f + 1) * T))
    g = torch.Generator().manual_seed(wl.seed + 1000)
    rows.update(torch.randperm(n, generator=g)[:n_random].tolist())
    return sorted(rows)


def sample_heads(wl: Workload) -> list:
    """(b, h) pairs whose rows are checked row by row at full size."""
    if wl.name == "sr_long":
        hs = sorted({0, wl.heads // 2 - 1, wl.heads - 1, *wl.boost_heads})
        return [(b, h) for b in range(wl.batch) for h in hs]
    if wl.name == "dense":
        hs = [0, wl.heads // 3, (2 * wl.heads) // 3, wl.heads - 1]
        return [(b, h) for b in range(wl.batch) for h in hs]
    return [(b, h) for b in range(wl.batch) for h in range(wl.heads)]


def micro(seed: int, batch: int, heads: int, head_dim: int, frames: int, ref_frames: int,
          tokens_per_frame: int, window: int, offset_std: float = 2.0):
    """Small random case with the same recipe, for brute-force pins."""
    wl = Workload("micro", batch, heads, head_dim, frames, ref_frames, tokens_per_frame,
                  window, seed)
    g = torch.Generator().manual_seed(seed)
    shape = (batch, heads, wl.n_tokens, head_dim)
    q = torch.randn(shape, generator=g)
    k = torch.randn(shape, generator=g)
    off = offset_std * torch.randn((heads, head_dim), generator=g)
    v = torch.randn(shape, generator=g)
    k += off[None, :, None, :]
    return wl, q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)
