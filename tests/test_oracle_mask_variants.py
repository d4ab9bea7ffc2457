"""Pins of the oracle's mask variants (CPU only).

The same mask family as the section "Deleting the mask" of the Google
Developers Blog post "HeyGen x Google Cloud: Bringing Avatar IV to TPUs"
(frames attend a window of nearby frames plus global reference frames),
with three variants the block-sparse method handles unchanged: a causal
window (frame f sees frames f - w .. f), reference frames after the video
frames in token order, and reference queries that see only reference keys.
Pinned by the pure-Python restatement (oracle.brute), closed-form counts of
active frame pairs, the relabelling invariance of the reference placement,
and brute-force attention and window bounds on tiny inputs.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from workloads import micro

VARIANTS = [0, 1, 2, 3, 4, 5, 6, 7]


def _kw(flags):
    return {"causal": bool(flags & 1), "ref_last": bool(flags & 2), "ref_local": bool(flags & 4)}


@pytest.mark.parametrize("flags", VARIANTS)
@pytest.mark.parametrize("F,T,w,R", [(4, 3, 1, 1), (5, 2, 2, 2), (3, 2, 0, 0), (4, 2, 5, 1)])
def test_mask_matches_python(flags, F, T, w, R):
    got = oracle.mask_dense(F, T, w, R, flags)
    want = np.array(brute.mask(F, T, w, R, **_kw(flags)), dtype=np.uint8)
    np.testing.assert_array_equal(got, want)


def _pairs_closed_form(F, w, R, flags):
    causal, local = flags & 1, flags & 4
    video = 0
    for f in range(F):
        lo = max(0, f - w)
        hi = f if causal else min(F - 1, f + w)
        video += (hi - lo + 1) + R           # video frames in the window, plus the references
    ref_rows = R * (R if local else F + R)  # reference queries
    return video + ref_rows


@pytest.mark.parametrize("flags", VARIANTS)
@pytest.mark.parametrize("F,w,R", [(21, 2, 1), (25, 3, 1), (13, 12, 1), (6, 0, 2), (9, 1, 0)])
def test_active_frame_pairs_closed_form(flags, F, w, R):
    bm = oracle.blockmap(F, 1, w, R, 1, 1, flags)  # one token per frame: blocks are frames
    assert bm["nnz"] == _pairs_closed_form(F, w, R, flags)
    assert bm["partial"] == 0


@pytest.mark.parametrize("flags", [0, 1, 4, 5])
def test_reference_suffix_is_a_relabelling(flags):
    # Moving the R reference frames from the front to the back permutes
    # tokens; outputs permute with them.
    F, T, w, R = 4, 16, 1, 1
    wl, q, k, v = micro(81, 1, 2, 16, F, R, T, w)
    n = (F + R) * T
    perm = np.concatenate([np.arange(R * T, n), np.arange(0, R * T)])  # suffix order -> prefix
    a = oracle.attention_full(q, k, v, F, T, w, R, wl.scale, flags)
    qs, ks, vs = (x[:, :, perm] for x in (q, k, v))
    b = oracle.attention_full(qs, ks, vs, F, T, w, R, wl.scale, flags | 2)
    np.testing.assert_allclose(b, a[:, perm], rtol=0, atol=1e-12)


@pytest.mark.parametrize("flags", VARIANTS)
def test_attention_matches_python_brute_force(flags):
    F, T, w, R = 3, 4, 1, 1
    wl, q, k, v = micro(82 + flags, 1, 1, 4, F, R, T, w)
    got = oracle.attention_full(q, k, v, F, T, w, R, wl.scale, flags)[0]
    want = brute.attention(q[0, 0].double().tolist(), k[0, 0].double().tolist(),
                           v[0, 0].double().tolist(), F, T, w, R, wl.scale, **_kw(flags))
    np.testing.assert_allclose(got, np.array(want), rtol=0, atol=1e-12)


@pytest.mark.parametrize("flags", [1, 2, 5, 7])
def test_window_bound_variants_match_python(flags):
    F, T, w, R = 4, 8, 1, 1
    wl, q, k, v = micro(90 + flags, 1, 1, 8, F, R, T, w)
    st = oracle.prepare_window(q, k, F, T, w, R, wl.scale, flags=flags)
    kh = k[0, 0].double().tolist()
    qh = q[0, 0].double().tolist()
    mu = brute.key_mean(kh)
    kn = [brute.norm([x - m for x, m in zip(row, mu)]) for row in kh]
    n = len(kh)
    for i in range(n):
        kw = max(kn[j] for j in range(n) if brute.attends(i, j, T, w, R, F=F, **_kw(flags)))
        assert st["b"][0, i] == pytest.approx(wl.scale * brute.norm(qh[i]) * kw, rel=1e-12)


def test_causal_first_frame_sees_only_itself_and_references():
    F, T, w, R = 5, 2, 2, 1
    m = oracle.mask_dense(F, T, w, R, 1)
    first_video = R * T
    row = m[first_video]
    assert row[:R * T].all() and row[R * T:(R + 1) * T].all()
    assert not row[(R + 1) * T:].any()
