"""Forward and window bounds under the mask variants (GPU).

wsattn_plan_ex(..., mask_flags) builds the block map of a variant of the
mask family (causal window, reference frames last, reference queries
local); the kernels run unchanged.  Outputs are compared with the oracle's
masked softmax of the same variant (max-abs 1e-2, relative L2 5e-3), the
window-bound statistics with oracle.prepare_window (relative 1e-5,
eligibility bit-exact).
"""
import numpy as np
import pytest
import torch

import oracle
from _helpers import TOL_MAX_ABS, TOL_REL_L2, flat_heads, gpu_run, rel_l2
from workloads import micro, sample_rows

pytestmark = pytest.mark.gpu


def _full_check(wl, q, k, v, out, flags):
    want = oracle.attention_full(q, k, v, wl.frames, wl.tokens_per_frame, wl.window,
                                 wl.ref_frames, wl.scale, flags)
    got = out.cpu().double().numpy().reshape(want.shape)
    assert np.abs(got - want).max() <= TOL_MAX_ABS
    assert rel_l2(got, want) <= TOL_REL_L2


@pytest.mark.parametrize("flags", [1, 2, 3, 4, 5, 6, 7])
def test_variant_forward_full_parity(flags):
    wl, q, k, v = micro(100 + flags, 1, 2, 128, 5, 1, 48, 1)
    _, out, _ = gpu_run(wl, q, k, v, mask_flags=flags)
    _full_check(wl, q, k, v, out, flags)


@pytest.mark.parametrize("flags", [1, 6])
def test_variant_forward_online_and_d64(flags):
    wl, q, k, v = micro(110 + flags, 2, 2, 64, 6, 2, 32, 2)
    _, out, _ = gpu_run(wl, q, k, v, mask_flags=flags, force_path=1)
    _full_check(wl, q, k, v, out, flags)
    _, out, _ = gpu_run(wl, q, k, v, mask_flags=flags)
    _full_check(wl, q, k, v, out, flags)


@pytest.mark.parametrize("case", range(8))
def test_random_shapes_full_parity(case):
    # seeded random shapes (tail sizes, windows, reference frames, mask
    # flags, head dims and block sizes), so merged tail tiles meet varied
    # groupings; both paths, every row against the oracle
    rng = np.random.default_rng(7000 + case)
    D = int(rng.choice([64, 128]))
    F = int(rng.integers(2, 9))
    R = int(rng.integers(0, 3))
    T = 16 * int(rng.integers(1, 21))
    w = int(rng.integers(0, 4))
    flags = int(rng.integers(0, 8))
    bk = int(rng.choice([b for b in range(16, min(T, 160) + 1, 16) if T % b == 0]))
    wl, q, k, v = micro(7000 + case, 1, 2, D, F, R, T, w)
    _, out, _ = gpu_run(wl, q, k, v, block_k=bk, mask_flags=flags)
    _full_check(wl, q, k, v, out, flags)
    _, out, _ = gpu_run(wl, q, k, v, block_k=bk, mask_flags=flags, force_path=1)
    _full_check(wl, q, k, v, out, flags)


@pytest.mark.parametrize("flags", [1, 3])
def test_variant_long_frames_sampled(flags):
    # SR frame span (T = 1040, 80-key blocks, 160-key steps) with a causal
    # window: each frame's keys are the reference run plus w + 1 frames.
    wl, q, k, v = micro(120 + flags, 1, 2, 128, 8, 1, 1040, 2)
    _, out, _ = gpu_run(wl, q, k, v, mask_flags=flags)
    rows = sample_rows(wl, n_random=64)
    pairs = [(h, r) for h in range(2) for r in rows]
    want = oracle.attention_rows(flat_heads(q, wl), flat_heads(k, wl), flat_heads(v, wl),
                                 wl.frames, wl.tokens_per_frame, wl.window, wl.ref_frames,
                                 wl.scale, pairs, flags).reshape(2, len(rows), wl.head_dim)
    got = flat_heads(out.cpu(), wl)[:, rows].double().numpy()
    assert np.abs(got - want).max() <= TOL_MAX_ABS
    assert rel_l2(got, want) <= TOL_REL_L2


@pytest.mark.parametrize("flags", [1, 2, 5, 7])
def test_variant_window_bounds(flags):
    import frame_aligned_window_gb300 as fw
    wl, q, k, v = micro(130 + flags, 1, 3, 128, 6, 1, 64, 1)
    plan, out, _ = gpu_run(wl, q, k, v, mask_flags=flags, bound=fw.BOUND_WINDOW)
    st = fw.wsattn_get_stats(plan, wl.batch)
    want = oracle.prepare_window(flat_heads(q, wl), flat_heads(k, wl), wl.frames,
                                 wl.tokens_per_frame, wl.window, wl.ref_frames, wl.scale,
                                 flags=flags)
    assert (np.abs(want["bmax"] - oracle.TAU) / oracle.TAU > 1e-3).all()
    np.testing.assert_array_equal(st["elig"], want["elig"])
    np.testing.assert_allclose(st["b"], want["b"], rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(st["bmax"], want["bmax"], rtol=1e-5)
    _full_check(wl, q, k, v, out, flags)
