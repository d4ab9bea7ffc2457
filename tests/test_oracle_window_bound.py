"""Pins of the oracle's window bound (oracle.prepare_window), CPU only.

The bound of the Google Developers Blog post "HeyGen x Google Cloud: Bringing
Avatar IV to TPUs", section "Breaking softmax's dependency chain", multiplies
a query's norm by a maximum key norm; any key set that holds the row's active
keys gives a valid bound.  The window variant takes the row's own active
keys.  Pinned here by:
  - a hand-worked case whose per-frame key norms are known in closed form;
  - a pure-Python brute force over the element mask (oracle.brute);
  - invariants: never above the global bound, equal to it for a dense mask,
    and every active centered logit at most the row's window bound.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from workloads import micro


def _frame_keys(values, T, d=2):
    """Keys [1, N, d]: every token of frame f is (values[f], 0, ...)."""
    k = torch.zeros(1, len(values) * T, d)
    for f, x in enumerate(values):
        k[0, f * T:(f + 1) * T, 0] = x
    return k.to(torch.bfloat16)


def test_hand_worked_window_bounds():
    # R = 1 reference frame with key value 3, video frames with values
    # 0..5, w = 1.  Mean 18/7; centered norms: reference 3/7, video
    # 18/7, 11/7, 4/7, 3/7, 10/7, 17/7.  Window maxima by frame (the
    # reference is in every window; reference rows see everything):
    #   ref 18/7, v0 18/7, v1 18/7, v2 11/7, v3 10/7, v4 17/7, v5 17/7.
    T, F, R, w = 16, 6, 1, 1
    k = _frame_keys([3, 0, 1, 2, 3, 4, 5], T)
    q = torch.zeros_like(k)
    q[..., 0] = 2.0  # ||q|| = 2
    scale = 1 / math.sqrt(2)
    st = oracle.prepare_window(q, k, F, T, w, R, scale)
    per_frame = np.array([18, 18, 18, 11, 10, 17, 17]) / 7
    want = scale * 2.0 * np.repeat(per_frame, T)
    np.testing.assert_allclose(st["b"][0], want, rtol=1e-13)
    np.testing.assert_allclose(st["kmax"][0], 18 / 7, rtol=1e-13)  # global maximum
    np.testing.assert_allclose(st["bmax"][0], scale * 2 * 18 / 7, rtol=1e-13)
    glob = oracle.prepare(q, k, scale)
    np.testing.assert_allclose(glob["b"][0], scale * 2 * 18 / 7, rtol=1e-13)


def test_window_bound_excludes_far_frame():
    # One far video frame carries large keys; rows whose window misses it
    # get a bound well below the global one, so a threshold between the two
    # separates the modes' eligibility.
    T, F, R, w = 16, 6, 0, 1
    k = _frame_keys([0, 0, 0, 0, 0, 12], T)
    q = torch.zeros_like(k)
    q[..., 0] = 1.0
    scale = 1.0
    st = oracle.prepare_window(q, k, F, T, w, R, scale, tau=5.0)
    glob = oracle.prepare(q, k, scale, tau=5.0)
    # mean 2: centered norms 2 for frames 0..4, 10 for frame 5
    per_frame = np.array([2, 2, 2, 2, 10, 10], dtype=float)
    np.testing.assert_allclose(st["b"][0], np.repeat(per_frame, T), rtol=1e-13)
    np.testing.assert_allclose(glob["b"][0], 10.0, rtol=1e-13)
    assert st["bmax"][0] == pytest.approx(10.0)
    # with frames 4, 5 excluded by a tighter window only frame 5's rows stay at 10
    st0 = oracle.prepare_window(q, k, F, T, 0, R, scale, tau=5.0)
    np.testing.assert_allclose(st0["b"][0], np.repeat([2, 2, 2, 2, 2, 10.0], T), rtol=1e-13)


@pytest.mark.parametrize("seed,F,R,T,w", [(61, 4, 1, 16, 1), (62, 5, 0, 16, 1), (63, 3, 2, 16, 0)])
def test_window_bound_matches_python_brute_force(seed, F, R, T, w):
    wl, q, k, v = micro(seed, 1, 2, 8, F, R, T, w)
    st = oracle.prepare_window(q, k, F, T, w, R, wl.scale)
    for h in range(2):
        kh = k[0, h].double().tolist()
        qh = q[0, h].double().tolist()
        mu = brute.key_mean(kh)
        kn = [brute.norm([x - m for x, m in zip(row, mu)]) for row in kh]
        n = len(kh)
        for i in range(n):
            kw = max(kn[j] for j in range(n) if brute.attends(i, j, T, w, R))
            assert st["b"][h, i] == pytest.approx(wl.scale * brute.norm(qh[i]) * kw, rel=1e-12)


@pytest.mark.parametrize("seed,F,R,T,w", [(64, 6, 1, 32, 1), (65, 7, 0, 16, 2), (66, 5, 1, 16, 9)])
def test_window_bound_invariants(seed, F, R, T, w):
    wl, q, k, v = micro(seed, 1, 3, 16, F, R, T, w)
    st = oracle.prepare_window(q, k, F, T, w, R, wl.scale)
    glob = oracle.prepare(q, k, wl.scale)
    assert (st["b"] <= glob["b"] * (1 + 1e-14)).all()
    np.testing.assert_array_equal(st["kmax"], glob["kmax"])
    if w >= F - 1:  # dense: every row sees every key
        np.testing.assert_allclose(st["b"], glob["b"], rtol=1e-14)
    m = oracle.mask_dense(F, T, w, R).astype(bool)
    qd = q[0].double().numpy()
    kd = k[0].double().numpy()
    for h in range(3):
        s = wl.scale * qd[h] @ (kd[h] - st["mu"][h]).T  # centered logits
        s = np.where(m, s, -np.inf)
        assert (s.max(axis=1) <= st["b"][h] * (1 + 1e-12) + 1e-12).all()
