"""Pins for the oracle's attention (CPU only).

The plain definition (masked softmax attention over the element mask) is
checked against an independent pure-Python brute force, a hand-worked
example, closed forms, a library routine (torch SDPA in fp64 for the dense
window) and the invariants the fixed-max method rests on (Google Developers
Blog post "HeyGen x Google Cloud: Bringing Avatar IV to TPUs", section
"Breaking softmax's dependency chain": centering is softmax-invariant, the
Cauchy-Schwarz bound holds for every key slice, and the fixed-max and
online-max formulations give the same result).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from workloads import WORKLOADS, generate, micro

MICRO = [
    # seed, B, H, D, F, R, T, w
    (11, 1, 2, 8, 3, 1, 4, 1),
    (12, 2, 1, 16, 4, 1, 3, 0),
    (13, 1, 1, 4, 5, 2, 2, 2),
    (14, 1, 3, 8, 2, 0, 5, 0),
    (15, 1, 1, 16, 4, 1, 16, 1),
]


def _lists(x):
    return x.to(torch.float64).tolist()


@pytest.mark.parametrize("case", MICRO)
def test_c_oracle_matches_python_brute_force(case):
    seed, B, H, D, F, R, T, w = case
    wl, q, k, v = micro(seed, B, H, D, F, R, T, w)
    got = oracle.attention_full(q, k, v, F, T, w, R, wl.scale)
    qf, kf, vf = (x.reshape(B * H, wl.n_tokens, D) for x in (q, k, v))
    for h in range(B * H):
        want = np.array(brute.attention(_lists(qf[h]), _lists(kf[h]), _lists(vf[h]), F, T, w, R,
                                        wl.scale))
        np.testing.assert_allclose(got[h], want, rtol=1e-12, atol=1e-13)


def test_hand_worked_example():
    # F=2 frames of T=2 tokens, no reference frame, w=0: each frame sees itself.
    # D=2, scale=1/sqrt(2).  Row 0: q=(3,4) against k0=(3,1), k1=(1,1):
    # logits 13/sqrt2 and 7/sqrt2 -> weight of v0 = 1/(1+exp(-6/sqrt2)).
    # Row 1: q=0 -> plain mean of v0, v1.
    q = torch.tensor([[3, 4], [0, 0], [1, 0], [0, -2]], dtype=torch.float64)
    k = torch.tensor([[3, 1], [1, 1], [3, 3], [1, 3]], dtype=torch.float64)
    v = torch.tensor([[1, 0], [0, 1], [2, 2], [-2, 4]], dtype=torch.float64)
    s = 1.0 / math.sqrt(2.0)
    out = oracle.attention_full(q[None], k[None], v[None], 2, 2, 0, 0, s)[0]
    sig = 1.0 / (1.0 + math.exp(-6.0 / math.sqrt(2.0)))
    np.testing.assert_allclose(out[0], [sig, 1 - sig], rtol=1e-14)
    np.testing.assert_allclose(out[1], [0.5, 0.5], rtol=1e-14)
    # row 2: q=(1,0) vs k2=(3,3), k3=(1,3): logits 3s, 1s -> weight 1/(1+e^{-2s})
    a = 1.0 / (1.0 + math.exp(-2.0 * s))
    np.testing.assert_allclose(out[2], [2 * a - 2 * (1 - a), 2 * a + 4 * (1 - a)], rtol=1e-14)
    # row 3: q=(0,-2): logits -6s, -6s -> equal weights
    np.testing.assert_allclose(out[3], [0.0, 3.0], atol=1e-14)


def test_zero_query_gives_mean_of_visible_values():
    wl, q, k, v = micro(21, 1, 2, 8, 4, 1, 3, 1)
    q = torch.zeros_like(q)
    F, T, w, R = wl.frames, wl.tokens_per_frame, wl.window, wl.ref_frames
    got = oracle.attention_full(q, k, v, F, T, w, R, wl.scale)
    m = np.array(brute.mask(F, T, w, R), dtype=np.float64)
    vf = v.to(torch.float64).reshape(2, wl.n_tokens, 8).numpy()
    for h in range(2):
        want = (m @ vf[h]) / m.sum(axis=1, keepdims=True)
        np.testing.assert_allclose(got[h], want, rtol=1e-12)


def test_constant_values_reproduced():
    wl, q, k, v = micro(22, 1, 1, 16, 5, 1, 4, 2)
    v = torch.full_like(v, 1.25)
    got = oracle.attention_full(q, k, v, wl.frames, wl.tokens_per_frame, wl.window,
                                wl.ref_frames, wl.scale)
    np.testing.assert_allclose(got, 1.25, rtol=1e-13)


def test_dense_window_equals_library_sdpa():
    # window >= F-1 makes the mask dense: plain softmax(q k^T * scale) v
    wl, q, k, v = micro(23, 1, 2, 16, 4, 1, 6, 3)
    got = oracle.attention_full(q, k, v, wl.frames, wl.tokens_per_frame, wl.window,
                                wl.ref_frames, wl.scale)
    qd, kd, vd = (x.to(torch.float64) for x in (q, k, v))
    want = torch.nn.functional.scaled_dot_product_attention(qd, kd, vd, scale=wl.scale)
    np.testing.assert_allclose(got, want.reshape(2, wl.n_tokens, 16).numpy(), rtol=1e-11,
                               atol=1e-13)


def test_centering_invariance():
    wl, q, k, v = micro(24, 1, 2, 16, 4, 1, 5, 1)
    F, T, w, R = wl.frames, wl.tokens_per_frame, wl.window, wl.ref_frames
    kd = k.to(torch.float64)
    mu = kd.mean(dim=2, keepdim=True)
    a = oracle.attention_full(q, kd, v, F, T, w, R, wl.scale)
    b = oracle.attention_full(q, kd - mu, v, F, T, w, R, wl.scale)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)
    # any other common shift too
    c = oracle.attention_full(q, kd + 3.5, v, F, T, w, R, wl.scale)
    np.testing.assert_allclose(a, c, rtol=1e-11, atol=1e-13)


@pytest.mark.parametrize("name", ["tiny"])
def test_every_logit_at_most_row_bound(name):
    wl = WORKLOADS[name]
    q, k, v = generate(wl)
    st = oracle.prepare(q, k, wl.scale)
    F, T, w, R = wl.frames, wl.tokens_per_frame, wl.window, wl.ref_frames
    m = oracle.mask_dense(F, T, w, R).astype(bool)
    qd, kd = oracle.as_f64(q), oracle.as_f64(k)
    for h in range(qd.shape[0]):
        kc = kd[h] - st["mu"][h]
        s = wl.scale * qd[h] @ kc.T
        s = np.where(m, s, -np.inf)
        assert (s.max(axis=1) <= st["b"][h] * (1 + 1e-12)).all()
        # the bound is attained by no row here, but is within a few units
        gap = st["b"][h] - s.max(axis=1)
        assert (gap >= 0).all()


@pytest.mark.parametrize("case", MICRO[:4])
def test_fixed_and_online_agree_with_plain(case):
    seed, B, H, D, F, R, T, w = case
    wl, q, k, v = micro(seed, B, H, D, F, R, T, w)
    st = oracle.prepare(q, k, wl.scale)
    pairs = [(h, i) for h in range(B * H) for i in range(wl.n_tokens)]
    plain = oracle.attention_rows(q, k, v, F, T, w, R, wl.scale, pairs)
    fixed = oracle.attention_rows_fixed(q, k, v, F, T, w, R, wl.scale, pairs, st)
    for bk in (1, T, 2 * T):
        online = oracle.attention_rows_online(q, k, v, F, T, w, R, wl.scale, bk, pairs)
        np.testing.assert_allclose(online, plain, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(fixed, plain, rtol=1e-12, atol=1e-14)


def test_fixed_and_online_agree_on_tiny_workload():
    wl = WORKLOADS["tiny"]
    q, k, v = generate(wl)
    st = oracle.prepare(q, k, wl.scale)
    F, T, w, R = wl.frames, wl.tokens_per_frame, wl.window, wl.ref_frames
    pairs = [(h, i) for h in range(wl.heads) for i in range(wl.n_tokens)]
    plain = oracle.attention_rows(q, k, v, F, T, w, R, wl.scale, pairs)
    fixed = oracle.attention_rows_fixed(q, k, v, F, T, w, R, wl.scale, pairs, st)
    online = oracle.attention_rows_online(q, k, v, F, T, w, R, wl.scale, 48, pairs)
    np.testing.assert_allclose(fixed, plain, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(online, plain, rtol=1e-12, atol=1e-14)


def test_row_subset_equals_full():
    wl, q, k, v = micro(25, 1, 2, 8, 3, 1, 4, 1)
    F, T, w, R = wl.frames, wl.tokens_per_frame, wl.window, wl.ref_frames
    full = oracle.attention_full(q, k, v, F, T, w, R, wl.scale)
    pairs = [(1, 7), (0, 0), (1, 15), (0, 9)]
    sub = oracle.attention_rows(q, k, v, F, T, w, R, wl.scale, pairs)
    for p, (h, i) in enumerate(pairs):
        np.testing.assert_array_equal(sub[p], full[h, i])
