"""Pure-Python brute force for tiny inputs.

TEST INFRASTRUCTURE ONLY (same rule as the rest of oracle/).  A second,
independent restatement of the definitions in the Google Developers Blog
post "HeyGen x Google Cloud: Bringing Avatar IV to TPUs" (section "Deleting
the mask" for the mask, section "Breaking softmax's dependency chain" for the
bound, section "Layout is ABI" for the pre-attention producer), written with
Python lists, loops and math.exp only, so that the C and numpy oracle can be
checked against it on tiny shapes.
"""
from __future__ import annotations

import math


def frame_of(tok: int, T: int) -> int:
    return tok // T


def attends(i: int, j: int, T: int, w: int, R: int, causal: bool = False,
            ref_last: bool = False, ref_local: bool = False, F: int = 0) -> bool:
    """Query token i sees key token j: key in a reference frame, or query in a
    reference frame, or the two video frames at most w apart.  Variants:
    causal (key frame at most w frames before, never after, the query's),
    ref_last (the R reference frames come after the F video frames; F is
    then needed), ref_local (reference queries see only reference keys)."""
    fi, fj = frame_of(i, T), frame_of(j, T)
    if ref_last:
        ref_i, ref_j, vi, vj = fi >= F, fj >= F, fi, fj
    else:
        ref_i, ref_j, vi, vj = fi < R, fj < R, fi - R, fj - R
    if ref_i:
        return ref_j if ref_local else True
    if ref_j:
        return True
    if causal:
        return 0 <= vi - vj <= w
    return abs(vi - vj) <= w


def mask(F: int, T: int, w: int, R: int, **variant):
    n = (F + R) * T
    return [[1 if attends(i, j, T, w, R, F=F, **variant) else 0 for j in range(n)]
            for i in range(n)]


def attention(q, k, v, F, T, w, R, scale, **variant):
    """q, k, v: nested lists [N][D] for one head.  Returns [N][D]."""
    n, d = len(q), len(q[0])
    out = []
    for i in range(n):
        logits = []
        for j in range(n):
            if attends(i, j, T, w, R, F=F, **variant):
                logits.append((j, scale * sum(q[i][c] * k[j][c] for c in range(d))))
        top = max(s for _, s in logits)
        weights = [(j, math.exp(s - top)) for j, s in logits]
        den = sum(e for _, e in weights)
        out.append([sum(e * v[j][c] for j, e in weights) / den for c in range(d)])
    return out


def key_mean(k):
    n, d = len(k), len(k[0])
    return [sum(k[j][c] for j in range(n)) / n for c in range(d)]


def norm(x):
    return math.sqrt(sum(t * t for t in x))


def produce(x, w, rope_cos, rope_sin, eps, heads, head_dim):
    """Pre-attention producer (section "Layout is ABI" of the same post:
    normalisation, projection, rotary embedding, head packing), restated with
    loops on nested lists.  x [B][N][C], w [3HD][C], rope tables [N][D/2].
    Returns (q, k, v) as nested lists [B][H][N][D]."""
    B, N, C = len(x), len(x[0]), len(x[0][0])
    H, D = heads, head_dim
    result = [[[[[0.0] * D for _ in range(N)] for _ in range(H)] for _ in range(B)]
              for _ in range(3)]
    for b in range(B):
        for t in range(N):
            ms = sum(val * val for val in x[b][t]) / C
            inv = 1.0 / math.sqrt(ms + eps)
            xh = [val * inv for val in x[b][t]]
            for part in range(3):
                for h in range(H):
                    feats = []
                    for d in range(D):
                        row = w[part * H * D + h * D + d]
                        feats.append(sum(row[c] * xh[c] for c in range(C)))
                    if part < 2:
                        for p in range(D // 2):
                            a, bb = feats[2 * p], feats[2 * p + 1]
                            co, si = rope_cos[t][p], rope_sin[t][p]
                            feats[2 * p] = a * co - bb * si
                            feats[2 * p + 1] = a * si + bb * co
                    result[part][b][h][t] = feats
    return result[0], result[1], result[2]
