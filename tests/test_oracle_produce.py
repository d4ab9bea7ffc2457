"""Pins of the pre-attention producer oracle (oracle.produce).

Google Developers Blog post "HeyGen x Google Cloud: Bringing Avatar IV to
TPUs", section "Layout is ABI", Figure 5: normalisation, rotary embedding,
projection and head packing, fused into one kernel that writes the
attention's input layout.  The oracle is checked against things other than
itself: the loop restatement in oracle/brute.py, closed forms of the RMS
normalisation, special rotation angles, the norm- and relative-position
invariants of a rotary embedding, and an identity projection that exposes
the head-packing order.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
import workloads


def _rand(seed, B, N, C, H, D):
    g = np.random.default_rng(seed)
    x = g.standard_normal((B, N, C)) * np.exp(0.5 * g.standard_normal((B, N, 1)))
    w = g.standard_normal((3 * H * D, C)) / math.sqrt(C)
    ang = g.uniform(-math.pi, math.pi, (N, D // 2))
    return x, w, np.cos(ang), np.sin(ang)


def test_matches_loop_restatement():
    B, N, C, H, D = 2, 5, 12, 2, 4
    x, w, c, s = _rand(1, B, N, C, H, D)
    q, k, v = oracle.produce(x, w, c, s, 1e-6, H, D)
    bq, bk, bv = brute.produce(x.tolist(), w.tolist(), c.tolist(), s.tolist(), 1e-6, H, D)
    np.testing.assert_allclose(q, np.array(bq), rtol=0, atol=1e-12)
    np.testing.assert_allclose(k, np.array(bk), rtol=0, atol=1e-12)
    np.testing.assert_allclose(v, np.array(bv), rtol=0, atol=1e-12)


def test_identity_projection_exposes_packing_and_normalisation():
    # C = 3 H D and W = I: before rotation the features are the normalised
    # token itself, q taking features [0, HD), k [HD, 2HD), v [2HD, 3HD),
    # head h its D consecutive features.
    B, N, H, D = 2, 3, 2, 4
    C = 3 * H * D
    x = np.arange(B * N * C, dtype=np.float64).reshape(B, N, C) % 7 - 3.0
    w = np.eye(C)
    ones, zeros = np.ones((N, D // 2)), np.zeros((N, D // 2))
    eps = 0.25
    q, k, v = oracle.produce(x, w, ones, zeros, eps, H, D)
    for b in range(B):
        for t in range(N):
            rms = math.sqrt(sum(val * val for val in x[b, t]) / C + eps)
            for h in range(H):
                for d in range(D):
                    assert q[b, h, t, d] == pytest.approx(x[b, t, h * D + d] / rms, abs=1e-14)
                    assert k[b, h, t, d] == pytest.approx(x[b, t, H * D + h * D + d] / rms,
                                                          abs=1e-14)
                    assert v[b, h, t, d] == pytest.approx(x[b, t, 2 * H * D + h * D + d] / rms,
                                                          abs=1e-14)


def test_constant_token_closed_form():
    # every feature of the token equals a: its normalised value is
    # a / sqrt(a^2 + eps)
    H, D, C = 1, 2, 6
    a, eps = 3.0, 1e-2
    x = np.full((1, 1, C), a)
    w = np.eye(C)
    q, k, v = oracle.produce(x, w, np.ones((1, 1)), np.zeros((1, 1)), eps, H, D)
    want = a / math.sqrt(a * a + eps)
    np.testing.assert_allclose(q.ravel(), [want, want], rtol=1e-15)
    np.testing.assert_allclose(v.ravel(), [want, want], rtol=1e-15)


def test_scale_invariance_without_eps():
    B, N, C, H, D = 1, 4, 16, 2, 4
    x, w, c, s = _rand(2, B, N, C, H, D)
    a = oracle.produce(x, w, c, s, 0.0, H, D)
    b = oracle.produce(x * 37.5, w, c, s, 0.0, H, D)
    for u, v in zip(a, b):
        np.testing.assert_allclose(u, v, rtol=1e-13, atol=1e-14)


def test_quarter_turn_and_no_turn():
    B, N, C, H, D = 1, 3, 8, 1, 4
    x, w, _, _ = _rand(3, B, N, C, H, D)
    ones, zeros = np.ones((N, D // 2)), np.zeros((N, D // 2))
    q0, k0, v0 = oracle.produce(x, w, ones, zeros, 1e-6, H, D)    # angle 0
    q1, k1, v1 = oracle.produce(x, w, zeros, ones, 1e-6, H, D)    # angle pi/2
    # (a, b) -> (-b, a): the sign and the pair order
    np.testing.assert_array_equal(q1[..., 0::2], -q0[..., 1::2])
    np.testing.assert_array_equal(q1[..., 1::2], q0[..., 0::2])
    np.testing.assert_array_equal(k1[..., 0::2], -k0[..., 1::2])
    np.testing.assert_array_equal(k1[..., 1::2], k0[..., 0::2])
    # v is never rotated
    np.testing.assert_array_equal(v0, v1)


def test_rotation_keeps_pair_norms():
    B, N, C, H, D = 2, 6, 16, 2, 8
    x, w, c, s = _rand(4, B, N, C, H, D)
    ones, zeros = np.ones((N, D // 2)), np.zeros((N, D // 2))
    q, k, _ = oracle.produce(x, w, c, s, 1e-6, H, D)
    q0, k0, _ = oracle.produce(x, w, ones, zeros, 1e-6, H, D)
    pn = lambda t: np.hypot(t[..., 0::2], t[..., 1::2])  # noqa: E731
    np.testing.assert_allclose(pn(q), pn(q0), rtol=1e-13)
    np.testing.assert_allclose(pn(k), pn(k0), rtol=1e-13)


def test_relative_position_property():
    # With angles position * freq_p (a 1-D rotary table), the logit of the
    # same query content at m and key content at n depends on m - n only.
    H, D, C, N = 1, 8, 16, 12
    g = np.random.default_rng(5)
    xq, xk = g.standard_normal(C), g.standard_normal(C)
    w = g.standard_normal((3 * H * D, C)) / math.sqrt(C)
    freq = 10000.0 ** (-np.arange(D // 2) / (D // 2))
    ang = np.arange(N)[:, None] * freq[None, :]
    c, s = np.cos(ang), np.sin(ang)

    def logit(m, n):
        x = np.zeros((1, N, C))
        x[0, m] = xq
        x[0, n] = xk if n != m else xq
        q, k, _ = oracle.produce(x, w, c, s, 1e-6, H, D)
        return float(q[0, 0, m] @ k[0, 0, n])

    for m, n, shift in ((2, 7, 3), (9, 1, 2), (4, 5, 6)):
        assert logit(m, n) == pytest.approx(logit(m + shift, n + shift), rel=1e-10, abs=1e-12)
    assert abs(logit(2, 7) - logit(2, 8)) > 1e-6  # and it does depend on m - n


def test_row_subset_matches_full():
    wl = workloads.Workload("p", 2, 2, 64, 2, 1, 16, 1, 9, grid_w=4)
    x, w, c, s = workloads.producer_inputs(wl)
    rows = [0, 5, 17, 47]
    full = oracle.produce(x, w, c, s, 1e-6, wl.heads, wl.head_dim)
    part = oracle.produce(x, w, c, s, 1e-6, wl.heads, wl.head_dim, rows=rows)
    for f, p in zip(full, part):
        np.testing.assert_array_equal(f[:, :, rows], p)


def test_inputs_recipe_shapes_and_table():
    wl = workloads.WORKLOADS["tiny"]
    x, w, c, s = workloads.producer_inputs(wl)
    assert x.dtype == torch.bfloat16 and x.shape == (1, wl.n_tokens, 128)
    assert w.shape == (3 * 128, 128)
    assert c.shape == (wl.n_tokens, 32) and c.dtype == torch.float32
    np.testing.assert_allclose((c.double() ** 2 + s.double() ** 2).numpy(), 1.0, atol=1e-6)
    assert torch.all(c[0] == 1) and torch.all(s[0] == 0)  # token 0: frame, row, col 0


def test_rope_table_decomposes_positions():
    # token -> (frame, row, column) of a frame's latent grid, each group of
    # dimension pairs turning by position * base^(-j / n)
    T, gw, D = 40, 8, 64
    c, s = workloads.rope_table(3 * T, T, gw, D)
    half = D // 2
    n_hw = half // 3
    n_t = half - 2 * n_hw
    tok = T + 2 * gw + 3                    # frame 1, row 2, column 3
    want = ([1 * 10000.0 ** (-j / n_t) for j in range(n_t)]
            + [2 * 10000.0 ** (-j / n_hw) for j in range(n_hw)]
            + [3 * 10000.0 ** (-j / n_hw) for j in range(n_hw)])
    np.testing.assert_allclose(c[tok].double().numpy(), np.cos(want), atol=1e-6)
    np.testing.assert_allclose(s[tok].double().numpy(), np.sin(want), atol=1e-6)
