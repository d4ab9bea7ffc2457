"""Pins for the oracle's mask and block classification (CPU only).

Source: Google Developers Blog post "HeyGen x Google Cloud: Bringing Avatar IV
to TPUs", section "Deleting the mask" and its Fig. 3.
"""
import itertools

import numpy as np
import pytest

import oracle
from oracle import brute
from workloads import WORKLOADS


def test_mask_matches_hand_derived_golden(golden):
    rows = golden("mask_F3_T2_R1_w1.txt")
    want = np.array([[int(c) for c in r] for r in rows], dtype=np.uint8)
    assert want.shape == (8, 8)
    np.testing.assert_array_equal(oracle.mask_dense(3, 2, 1, 1), want)
    np.testing.assert_array_equal(np.array(brute.mask(3, 2, 1, 1), dtype=np.uint8), want)


@pytest.mark.parametrize("F,T,w,R", [
    (1, 3, 0, 0), (2, 2, 0, 1), (4, 3, 1, 1), (5, 2, 2, 2), (5, 1, 0, 0), (3, 4, 5, 1),
    (6, 2, 1, 0), (4, 16, 1, 1),
])
def test_mask_c_matches_brute(F, T, w, R):
    np.testing.assert_array_equal(oracle.mask_dense(F, T, w, R),
                                  np.array(brute.mask(F, T, w, R), dtype=np.uint8))


def test_mask_properties():
    # reference columns always active; reference rows dense; video block is
    # symmetric and banded with half-width w (frame granularity)
    F, T, w, R = 6, 3, 2, 1
    m = oracle.mask_dense(F, T, w, R)
    assert m[:, :R * T].all() and m[:R * T, :].all()
    np.testing.assert_array_equal(m, m.T)
    fr = m[R * T::T, R * T::T]
    for f, g in itertools.product(range(F), range(F)):
        assert fr[f, g] == (abs(f - g) <= w)


def test_frame_pair_counts_hand_count(golden):
    for line in golden("frame_pairs.txt"):
        name, F, R, w, pairs = line.split()
        F, R, w, pairs = int(F), int(R), int(w), int(pairs)
        wl = WORKLOADS[name]
        assert (wl.frames, wl.ref_frames, wl.window) == (F, R, w)
        # frame-granular block map: one block per frame
        bm = oracle.blockmap(F, 1, w, R, 1, 1)
        assert bm["nnz"] == pairs and bm["partial"] == 0


def test_tiny_active_element_count(golden):
    wl = WORKLOADS["tiny"]
    m = oracle.mask_dense(wl.frames, wl.tokens_per_frame, wl.window, wl.ref_frames)
    assert int(m.sum()) == 19 * wl.tokens_per_frame ** 2


def valid_blocks(T):
    return [b for b in range(16, T + 1, 16) if T % b == 0]


@pytest.mark.parametrize("name", ["tiny", "small"])
def test_blockmap_all_valid_sizes_full_or_empty(name):
    wl = WORKLOADS[name]
    F, T, w, R = wl.frames, wl.tokens_per_frame, wl.window, wl.ref_frames
    pairs = oracle.blockmap(F, 1, w, R, 1, 1)["nnz"]
    m = oracle.mask_dense(F, T, w, R)
    for bq, bk in itertools.product(valid_blocks(T), valid_blocks(T)):
        bm = oracle.blockmap(F, T, w, R, bq, bk)
        assert bm["partial"] == 0
        assert bm["nnz"] == pairs * (T // bq) * (T // bk)
        n = m.shape[0]
        anyb = m.reshape(n // bq, bq, n // bk, bk).any(axis=(1, 3))
        np.testing.assert_array_equal(bm["bitmap"].astype(bool), anyb)


def test_blockmap_sr_shaped_auto_size():
    wl = WORKLOADS["sr"]
    bm = oracle.blockmap(wl.frames, wl.tokens_per_frame, wl.window, wl.ref_frames, 80, 80)
    assert bm["partial"] == 0 and bm["nnz"] == 142 * 13 * 13


def test_blockmap_detects_partial_blocks():
    # a block size that does not divide the frame span straddles frame edges
    F, T, w, R = 5, 24, 1, 1  # N = 144 = 9 * 16, but 16 does not divide T
    bm = oracle.blockmap(F, T, w, R, 16, 16)
    assert bm["partial"] > 0
    m = oracle.mask_dense(F, T, w, R)
    n = m.shape[0]
    blk = m.reshape(n // 16, 16, n // 16, 16).sum(axis=(1, 3))
    assert bm["partial"] == int(((blk > 0) & (blk < 256)).sum())
    assert bm["full"] == int((blk == 256).sum())


def test_blockmap_csr_order():
    bm = oracle.blockmap(5, 32, 1, 1, 16, 32)
    rp, col = bm["row_ptr"], bm["col"]
    for r in range(len(rp) - 1):
        row = col[rp[r]:rp[r + 1]]
        assert list(row) == sorted(row)
        np.testing.assert_array_equal(np.flatnonzero(bm["bitmap"][r]), row)
