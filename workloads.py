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

The pre-attention producer takes hidden states x [B, N, C], projection
weights W [3 H D, C] and a rotary angle table (cos, sin) [N, D / 2]; the
table is an input that encodes each token's position (frame, row, column of
the latent grid), built here like any other input (`producer_inputs`).
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
    grid_w: int = 0          # columns of a frame's latent grid (0: one row of T)

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
    "tiny": Workload("tiny", 1, 2, 64, 4, 1, 48, 1, 0, grid_w=8,
                     description="4 frames + 1 reference, 48 tokens/frame"),
    "small": Workload("small", 1, 8, 128, 9, 1, 208, 1, 1, grid_w=16,
                      description="9 frames + 1 reference, 13x16 tokens/frame"),
    "sr": Workload("sr", 1, 24, 128, 21, 1, 1040, 2, 2, grid_w=40,
                   description="SR-shaped: 21 frames + 1 reference, 26x40 latent grid"),
    "sr_long": Workload("sr_long", 1, 24, 128, 25, 1, 2080, 3, 3, boost_heads=(5, 17),
                        grid_w=40,
                        description="SR-long: 25 frames + 1 reference; heads 5 and 17 "
                                    "have 1% of query rows scaled x8"),
    "dense": Workload("dense", 2, 40, 128, 13, 1, 1568, 12, 4, grid_w=56,
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


def rope_table(n_tokens: int, tokens_per_frame: int, grid_w: int, head_dim: int,
               base: float = 10000.0):
    """Rotary angle table (cos, sin), fp32 [N, D / 2], for tokens laid out as
    frames of a latent grid grid_w columns wide: the D / 2 dimension pairs are
    split into a frame group (the remainder), a row group and a column group
    (floor(D / 6) pairs each); pair j of a group of n pairs turns by
    position * base^(-j / n)."""
    half = head_dim // 2
    n_hw = half // 3
    n_t = half - 2 * n_hw
    gw = grid_w if grid_w > 0 else tokens_per_frame
    tok = torch.arange(n_tokens, dtype=torch.float64)
    frame = torch.div(tok, tokens_per_frame, rounding_mode="floor")
    inner = tok - frame * tokens_per_frame
    row = torch.div(inner, gw, rounding_mode="floor")
    col = inner - row * gw
    parts = []
    for pos, n in ((frame, n_t), (row, n_hw), (col, n_hw)):
        freq = base ** (-torch.arange(n, dtype=torch.float64) / n)
        parts.append(pos[:, None] * freq[None, :])
    ang = torch.cat(parts, dim=1)
    return torch.cos(ang).to(torch.float32).contiguous(), torch.sin(ang).to(torch.float32).contiguous()


def producer_inputs(wl: Workload, model_dim: int = 0, seed_offset: int = 500):
    """(x, w, rope_cos, rope_sin) for the pre-attention producer of wl.

    C = model_dim or H * D.  Draw order from one torch CPU generator seeded
    with wl.seed + seed_offset: m [C] (a component every token shares, so the
    projected keys of a head share one too), z [B, N, C], per-token scales
    exp(0.5 * N(0, 1)) (so the normalisation matters), W [3 H D, C] / sqrt(C).
    x = (z + m) * scale, cast to bf16; W cast to bf16."""
    C = model_dim or wl.heads * wl.head_dim
    g = torch.Generator().manual_seed(wl.seed + seed_offset)
    m = torch.randn(C, generator=g)
    z = torch.randn((wl.batch, wl.n_tokens, C), generator=g)
    sc = torch.exp(0.5 * torch.randn((wl.batch, wl.n_tokens, 1), generator=g))
    w = torch.randn((3 * wl.heads * wl.head_dim, C), generator=g) / float(C) ** 0.5
    x = ((z + m) * sc).to(torch.bfloat16).contiguous()
    cos, sin = rope_table(wl.n_tokens, wl.tokens_per_frame, wl.grid_w, wl.head_dim)
    return x, w.to(torch.bfloat16).contiguous(), cos, sin
