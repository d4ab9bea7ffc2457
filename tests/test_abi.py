"""The C ABI on the CPU: the library loads, exports every declared symbol, and
its host-side plan (block map, CSR, work list geometry, argument checks) is
bit-exact against the oracle's element-by-element classification."""
import ctypes
import itertools
import os
import re

import numpy as np
import pytest
import torch

import oracle
from workloads import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    with open(os.path.join(ROOT, "include", "wsattn.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^(?:int|const char\*)\s+(wsattn_\w+)\(", text, re.M)))


def test_library_exports_every_declared_symbol():
    import frame_aligned_window_gb300 as fw
    lib = ctypes.CDLL(fw.LIB_PATH)
    declared = _declared_symbols()
    assert len(declared) >= 12
    assert set(declared) == set(fw.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings():
    import frame_aligned_window_gb300 as fw
    for code in range(9):
        assert fw.wsattn_status_string(code) and fw.wsattn_status_string(code) != "unknown status"
    assert fw.wsattn_status_string(99) == "unknown status"


def valid_blocks(T, cap=None):
    return [b for b in range(16, (cap or T) + 1, 16) if T % b == 0]


def _plan_vs_oracle(F, T, w, R, bq, bk, flags=0):
    import frame_aligned_window_gb300 as fw
    plan = fw.wsattn_plan(F, T, w, R, 2, 128, bq, bk, flags)
    want = oracle.blockmap(F, T, w, R, bq, bk, flags)
    assert want["partial"] == 0
    np.testing.assert_array_equal(fw.wsattn_get_block_map(plan), want["bitmap"])
    rp, col = fw.wsattn_get_csr(plan)
    np.testing.assert_array_equal(rp, want["row_ptr"])
    np.testing.assert_array_equal(col, want["col"])
    assert plan.nnz == want["nnz"]
    m_pairs = oracle.blockmap(F, T, w, R, T, T, flags)["nnz"] * T * T
    assert plan.active_pairs == m_pairs
    _check_work_list(plan, F, T, w, R, bk, flags)
    plan.destroy()


def _runs_set(run0, len0, run1, len1):
    return set(range(run0, run0 + len0)) | set(range(run1, run1 + len1))


def _check_work_list(plan, F, T, w, R, bk, flags=0):
    """The forward work list against the oracle's frame-level block map
    (query block = one frame): every query token lies in exactly one tile
    row, and each row's own key blocks are its frame's.  A merged tail tile
    (gsz > 0) walks the union of its row groups' blocks."""
    import frame_aligned_window_gb300 as fw
    tiles, groups = fw.wsattn_get_tiles(plan)
    assert len(tiles) == plan.tiles_per_head
    frame_keys = oracle.blockmap(F, T, w, R, T, bk, flags)["bitmap"]  # [F+R, N/bk]
    N = (F + R) * T
    seen = np.zeros(N, dtype=np.int32)
    tail = T % 128
    n_merged = 0
    for row0, nvalid, nblk, run0, len0, run1, nstep, kbeg, gsz, gtab in tiles:
        assert 0 < nvalid <= 128 and nblk == len0 + (nblk - len0) and nstep > 0
        walk = _runs_set(run0, len0, run1, nblk - len0)
        assert len(walk) == nblk
        if gsz == 0:
            toks = np.arange(row0, row0 + nvalid)
            frames = toks // T
            assert (frames == frames[0]).all()
            want = set(np.flatnonzero(frame_keys[frames[0]]))
            assert walk == want, (row0, nvalid)
        else:
            n_merged += 1
            assert gsz == tail and nvalid % gsz == 0 and nvalid // gsz >= 2
            union = set()
            toks = []
            for i in range(nvalid // gsz):
                g = groups[gtab + i]
                own = _runs_set(*g)
                t0 = row0 + i * T
                f = t0 // T
                assert (t0 + gsz - 1) // T == f and (t0 % T) == T - tail
                assert own == set(np.flatnonzero(frame_keys[f])), (row0, i)
                union |= own
                toks.extend(range(t0, t0 + gsz))
            assert walk == union
            toks = np.array(toks)
        seen[toks] += 1
    assert (seen == 1).all()
    if tail == 0:
        assert n_merged == 0 and plan.tiles_per_head == (F + R) * (T // 128)
    else:
        assert plan.tiles_per_head <= (F + R) * ((T + 127) // 128)


@pytest.mark.parametrize("name", ["sr", "sr_long", "dense"])
def test_work_list_merges_frame_tails(name):
    # T mod 128 = 16 (SR) or 32 (SR-long, dense): consecutive frames' tails
    # share tiles, and every row still walks exactly its frame's key blocks
    import frame_aligned_window_gb300 as fw
    wl = WORKLOADS[name]
    plan = fw.wsattn_plan(wl.frames, wl.tokens_per_frame, wl.window, wl.ref_frames, wl.heads,
                          wl.head_dim)
    _check_work_list(plan, wl.frames, wl.tokens_per_frame, wl.window, wl.ref_frames,
                     plan.block_k)
    tiles, groups = fw.wsattn_get_tiles(plan)
    assert (tiles[:, 8] > 0).any() and len(groups) > 0
    plan.destroy()


def test_work_list_random_shapes():
    # seeded random shapes: frame counts, token spans with every tail size
    # (T mod 128 in 16 .. 112, or none), windows, reference frames, all
    # mask flags and random valid block sizes; the work list must cover each
    # token once with its own frame's key blocks
    import frame_aligned_window_gb300 as fw
    rng = np.random.default_rng(20261202)
    for _ in range(60):
        F = int(rng.integers(1, 14))
        R = int(rng.integers(0, 3))
        T = 16 * int(rng.integers(1, 30))
        w = int(rng.integers(0, 5))
        flags = int(rng.integers(0, 8))
        blocks = valid_blocks(T, 160)
        bk = int(rng.choice(blocks))
        plan = fw.wsattn_plan(F, T, w, R, 2, 128, 0, bk, flags)
        _check_work_list(plan, F, T, w, R, bk, flags)
        plan.destroy()


def test_get_tiles_checks_capacities():
    import frame_aligned_window_gb300 as fw
    wl = WORKLOADS["sr"]
    plan = fw.wsattn_plan(wl.frames, wl.tokens_per_frame, wl.window, wl.ref_frames, wl.heads,
                          wl.head_dim)
    tiles, groups = fw.wsattn_get_tiles(plan)
    fn = fw.raw_call("wsattn_get_tiles")
    t = np.zeros(tiles.size, dtype=np.int32)
    g = np.zeros(groups.size, dtype=np.int32)
    tp, gp = ctypes.c_void_p(t.ctypes.data), ctypes.c_void_p(g.ctypes.data)
    assert fn(plan.handle, tp, t.size, gp, g.size) == 0
    np.testing.assert_array_equal(t.reshape(tiles.shape), tiles)
    np.testing.assert_array_equal(g.reshape(groups.shape), groups)
    assert fn(plan.handle, tp, t.size - 1, gp, g.size) == 1   # one int short: BAD_ARG
    assert fn(plan.handle, tp, t.size, gp, g.size - 1) == 1
    assert fn(plan.handle, None, t.size, gp, g.size) == 1
    assert fn(plan.handle, tp, t.size, None, g.size) == 1
    assert fn(None, tp, t.size, gp, g.size) == 1
    plan.destroy()
    # no merged tiles (T a multiple of 128): an empty group table, NULL allowed
    plan = fw.wsattn_plan(3, 256, 1, 1, 2, 128)
    tiles, groups = fw.wsattn_get_tiles(plan)
    assert len(groups) == 0 and (tiles[:, 8] == 0).all() and len(tiles) == 4 * 2
    t = np.zeros(tiles.size, dtype=np.int32)
    assert fn(plan.handle, ctypes.c_void_p(t.ctypes.data), t.size, None, 0) == 0
    plan.destroy()


@pytest.mark.parametrize("name", ["tiny", "small"])
def test_plan_matches_oracle_all_valid_sizes(name):
    wl = WORKLOADS[name]
    T = wl.tokens_per_frame
    for bq, bk in itertools.product(valid_blocks(T), valid_blocks(T)):
        _plan_vs_oracle(wl.frames, T, wl.window, wl.ref_frames, bq, bk)


@pytest.mark.parametrize("flags", [1, 2, 3, 4, 5, 6, 7])
@pytest.mark.parametrize("F,T,w,R,bq,bk", [(4, 48, 1, 1, 16, 48), (7, 32, 2, 2, 32, 16),
                                           (5, 16, 9, 1, 16, 16), (6, 32, 0, 0, 32, 32)])
def test_plan_matches_oracle_mask_variants(flags, F, T, w, R, bq, bk):
    _plan_vs_oracle(F, T, w, R, bq, bk, flags)


def test_plan_rejects_unknown_mask_flags():
    import frame_aligned_window_gb300 as fw
    with pytest.raises(fw.WsattnError) as e:
        fw.wsattn_plan(4, 48, 1, 1, 2, 64, 0, 0, 8)
    assert e.value.code == 1


@pytest.mark.parametrize("bq,bk", [(80, 80), (16, 208), (1040, 80), (208, 16)])
def test_plan_matches_oracle_sr_shaped(bq, bk):
    wl = WORKLOADS["sr"]
    _plan_vs_oracle(wl.frames, wl.tokens_per_frame, wl.window, wl.ref_frames, bq, bk)


@pytest.mark.parametrize("case", [
    (1, 16, 0, 0, 16, 16), (3, 32, 0, 2, 16, 32), (6, 48, 10, 1, 48, 16), (5, 64, 1, 0, 32, 64),
    (2, 160, 1, 1, 160, 160),
])
def test_plan_matches_oracle_edge_shapes(case):
    _plan_vs_oracle(*case)


def test_auto_block_sizes():
    import frame_aligned_window_gb300 as fw
    # longest forward step floor(160 / bk) * bk, larger bk on ties
    expect = {"tiny": 16, "small": 16, "sr": 80, "sr_long": 160, "dense": 32}
    for name, bk in expect.items():
        wl = WORKLOADS[name]
        plan = fw.wsattn_plan(wl.frames, wl.tokens_per_frame, wl.window, wl.ref_frames,
                              wl.heads, wl.head_dim)
        assert (plan.block_q, plan.block_k) == (bk, bk), name
        assert plan.n_tokens == wl.n_tokens


def test_plan_errors():
    import frame_aligned_window_gb300 as fw
    bad = [
        ((0, 48, 1, 1, 2, 64, 0, 0), 1),     # no frames
        ((4, 48, -1, 1, 2, 64, 0, 0), 1),    # negative window
        ((4, 48, 1, -1, 2, 64, 0, 0), 1),    # negative ref frames
        ((4, 48, 1, 1, 0, 64, 0, 0), 1),     # no heads
        ((4, 40, 1, 1, 2, 64, 0, 0), 2),     # T not a multiple of 16
        ((4, 48, 1, 1, 2, 64, 32, 0), 2),    # 32 does not divide 48
        ((4, 48, 1, 1, 2, 64, 0, 24), 2),    # not a multiple of 16
        ((4, 48, 1, 1, 2, 96, 0, 0), 3),     # head_dim
    ]
    for args, code in bad:
        with pytest.raises(fw.WsattnError) as e:
            fw.wsattn_plan(*args)
        assert e.value.code == code, args
    h = ctypes.c_void_p()
    assert fw.raw_call("wsattn_plan")(4, 48, 1, 1, 2, 64, 0, 0, None) == 1
    assert fw.raw_call("wsattn_plan")(4, 48, 1, 1, 2, 64, 0, 0, ctypes.byref(h)) == 0
    assert fw.raw_call("wsattn_plan_destroy")(h) == 0
    assert fw.raw_call("wsattn_plan_destroy")(None) == 0


def test_call_order_errors_without_device_work():
    import frame_aligned_window_gb300 as fw
    plan = fw.wsattn_plan(4, 48, 1, 1, 2, 64)
    fwd = fw.raw_call("wsattn_forward")
    dummy = ctypes.c_void_p(1 << 20)  # aligned, never dereferenced: the checks come first
    assert fwd(plan.handle, 1, dummy, dummy, dummy, dummy, None) == 4   # NOT_PREPARED
    assert fwd(plan.handle, 0, dummy, dummy, dummy, dummy, None) == 1   # batch 0
    assert fwd(plan.handle, 1, None, dummy, dummy, dummy, None) == 1    # null q
    prep = fw.raw_call("wsattn_prepare")
    assert prep(plan.handle, 0, dummy, dummy, None) == 1
    assert prep(plan.handle, 1, ctypes.c_void_p((1 << 20) + 2), dummy, None) == 1  # misaligned
    stats = fw.raw_call("wsattn_get_stats")
    assert stats(plan.handle, None, None, None, None, None, None, None) == 4
    assert fw.raw_call("wsattn_plan_set_debug")(plan.handle, 2, ctypes.c_float(0.0)) == 1
    assert fw.raw_call("wsattn_device_status")(plan.handle, None) == 0  # no device work yet
    small = (ctypes.c_uint8 * 4)()
    assert fw.raw_call("wsattn_get_block_map")(plan.handle, small, 4) == 1


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU failure path")
def test_prepare_without_gpu_fails_loudly():
    import frame_aligned_window_gb300 as fw
    plan = fw.wsattn_plan(4, 48, 1, 1, 2, 64)
    dummy = ctypes.c_void_p(1 << 20)
    assert fw.raw_call("wsattn_prepare")(plan.handle, 1, dummy, dummy, None) == 6  # CUDA


def test_produce_argument_errors_without_device_work():
    # wsattn_produce checks every argument before any CUDA call
    import frame_aligned_window_gb300 as fw
    produce = fw.raw_call("wsattn_produce")
    a = ctypes.c_void_p(1 << 20)            # aligned, never dereferenced
    mis = ctypes.c_void_p((1 << 20) + 8)    # not 16-byte aligned
    f = ctypes.c_float
    plan = fw.wsattn_plan(4, 48, 1, 1, 2, 128)      # H * D = 256
    ok_args = [plan.handle, 1, a, 256, a, a, a, f(1e-6), a, a, a, None]

    def call(**over):
        args = list(ok_args)
        names = ["plan", "batch", "x", "c", "w", "cos", "sin", "eps", "q", "k", "v", "stream"]
        for key, val in over.items():
            args[names.index(key)] = val
        return produce(*args)

    assert call(batch=0) == 1
    for key in ("x", "w", "cos", "sin", "q", "k", "v"):
        assert call(**{key: None}) == 1, key
        assert call(**{key: mis}) == 1, key
    assert call(c=96) == 1            # not a multiple of 64
    assert call(c=0) == 1
    assert call(eps=f(-1.0)) == 1
    assert call(eps=f(float("nan"))) == 1
    assert call(eps=f(float("inf"))) == 1
    assert call(plan=None) == 1
    # H * D = 64 is not a multiple of 128
    small = fw.wsattn_plan(4, 48, 1, 1, 1, 64)
    assert produce(small.handle, 1, a, 64, a, a, a, f(1e-6), a, a, a, None) == 3


def test_release_library_reports_no_debug_flag():
    import frame_aligned_window_gb300 as fw
    if os.environ.get("WSATTN_LIBRARY"):
        pytest.skip("another build of the library is loaded")
    assert fw.wsattn_build_flags() == 0
    assert fw.wsattn_status_string(9) == "device bounds check failed (debug build)"
