"""Window row bounds (wsattn_plan_set_bound(WINDOW)) vs the oracle (GPU).

The statistics are compared like the global ones (fp32 reductions of exact
bf16 inputs against fp64: relative 1e-5; eligibility bit-exact away from
tau), and forward outputs like every other forward test (max-abs 1e-2,
relative L2 5e-3).
"""
import numpy as np
import pytest
import torch

import oracle
from _helpers import flat_heads, oracle_rows, rel_l2, workload
from workloads import generate, micro, sample_rows

pytestmark = pytest.mark.gpu

REL_BOUND = 1e-5
TOL_MAX_ABS, TOL_REL_L2 = 1e-2, 5e-3


def _window_stats_gpu(wl, q, k, tau=0.0):
    import frame_aligned_window_gb300 as fw
    plan = fw.wsattn_plan(wl.frames, wl.tokens_per_frame, wl.window, wl.ref_frames, wl.heads,
                          wl.head_dim)
    if tau > 0:
        fw.wsattn_plan_set_debug(plan, -1, tau)
    fw.wsattn_plan_set_bound(plan, fw.BOUND_WINDOW)
    qd, kd = q.cuda(), k.cuda()
    fw.wsattn_prepare(plan, qd, kd)
    st = fw.wsattn_get_stats(plan, wl.batch)
    assert fw.wsattn_device_status(plan) == 0
    return plan, qd, kd, st


@pytest.mark.parametrize("name,heads", [("tiny", None), ("small", None), ("sr", [0, 23])])
def test_window_stats_match_oracle(name, heads):
    wl = workload(name)
    q, k, v = generate(wl)
    _, _, _, st = _window_stats_gpu(wl, q, k)
    qf, kf = flat_heads(q, wl), flat_heads(k, wl)
    sel = list(range(qf.shape[0])) if heads is None else heads
    want = oracle.prepare_window(qf[sel], kf[sel], wl.frames, wl.tokens_per_frame, wl.window,
                                 wl.ref_frames, wl.scale)
    assert (np.abs(want["bmax"] - oracle.TAU) / oracle.TAU > 1e-3).all()
    np.testing.assert_array_equal(st["elig"][sel], want["elig"])
    np.testing.assert_allclose(st["kmax"][sel], want["kmax"], rtol=REL_BOUND)
    np.testing.assert_allclose(st["bmax"][sel], want["bmax"], rtol=REL_BOUND)
    np.testing.assert_allclose(st["b"][sel], want["b"], rtol=REL_BOUND, atol=1e-6)
    np.testing.assert_array_equal(st["bmax"], st["b"].max(axis=1))
    qd64 = qf[sel].double().numpy()
    c = wl.scale * np.einsum("hnd,hd->hn", qd64, want["mu"])
    np.testing.assert_allclose(st["m"][sel], want["b"] + c, rtol=0,
                               atol=1e-5 * (1 + np.abs(want["b"] + c).max()))
    # never above the global bound of the same head
    glob = oracle.prepare(qf[sel], kf[sel], wl.scale)
    assert (st["b"][sel] <= glob["b"] * (1 + 1e-5) + 1e-6).all()


def _far_frame_case():
    # Frame 5 carries large keys; the queries of frames 4 and 5 (the only
    # ones whose window holds frame 5) are zero.  The global bound of every
    # other row then uses frame 5's norm, the window bound does not.
    wl, q, k, v = micro(71, 1, 2, 128, 6, 0, 48, 1)
    T = wl.tokens_per_frame
    k = k.float()
    k[:, :, 5 * T:6 * T] *= 6.0
    k = k.to(torch.bfloat16)
    q = q.clone()
    q[:, :, 4 * T:6 * T] = 0
    return wl, q, k, v


def test_window_bound_flips_eligibility_and_forward_matches():
    import frame_aligned_window_gb300 as fw
    wl, q, k, v = _far_frame_case()
    qf, kf = flat_heads(q, wl), flat_heads(k, wl)
    glob = oracle.prepare(qf, kf, wl.scale)
    win = oracle.prepare_window(qf, kf, wl.frames, wl.tokens_per_frame, wl.window,
                                wl.ref_frames, wl.scale)
    assert (win["bmax"] < 0.6 * glob["bmax"]).all()
    tau = float(np.sqrt(win["bmax"].max() * glob["bmax"].min()))  # between the two
    assert (np.abs(win["bmax"] - tau) / tau > 1e-3).all()
    assert (np.abs(glob["bmax"] - tau) / tau > 1e-3).all()
    plan, qd, kd, st = _window_stats_gpu(wl, q, k, tau=tau)
    assert st["elig"].all()
    vd = v.cuda()
    out = fw.wsattn_forward(plan, qd, kd, vd)
    torch.cuda.synchronize()
    assert fw.wsattn_device_status(plan) == 0
    # the same plan in global mode: every head ineligible (online path)
    fw.wsattn_plan_set_bound(plan, fw.BOUND_GLOBAL)
    fw.wsattn_prepare(plan, qd, kd)
    st_g = fw.wsattn_get_stats(plan, wl.batch)
    assert not st_g["elig"].any()
    out_g = fw.wsattn_forward(plan, qd, kd, vd)
    torch.cuda.synchronize()
    want = oracle.attention_full(q, k, v, wl.frames, wl.tokens_per_frame, wl.window,
                                 wl.ref_frames, wl.scale)
    for o in (out, out_g):
        got = o.cpu().double().numpy().reshape(want.shape)
        assert np.abs(got - want).max() <= TOL_MAX_ABS
        assert rel_l2(got, want) <= TOL_REL_L2


def test_window_forward_matches_oracle_sr_long_sampled():
    import frame_aligned_window_gb300 as fw
    wl = workload("sr_long")
    q, k, v = generate(wl)
    plan, qd, kd, st = _window_stats_gpu(wl, q, k)
    out = fw.wsattn_forward(plan, qd, kd, v.cuda())
    torch.cuda.synchronize()
    assert fw.wsattn_device_status(plan) == 0
    bh = [(0, 0), (0, 5), (0, 17)]
    rows = sample_rows(wl, n_random=64)
    want = oracle_rows(wl, q, k, v, bh, rows)
    got = torch.stack([out[b, h, rows] for b, h in bh]).cpu().double().numpy()
    assert np.abs(got - want.reshape(got.shape)).max() <= TOL_MAX_ABS
    assert rel_l2(got, want.reshape(got.shape)) <= TOL_REL_L2


def test_set_bound_requires_prepare_and_checks_mode():
    import frame_aligned_window_gb300 as fw
    wl, q, k, v = micro(72, 1, 2, 64, 3, 1, 48, 1)
    plan = fw.wsattn_plan(wl.frames, wl.tokens_per_frame, wl.window, wl.ref_frames, wl.heads,
                          wl.head_dim)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    fw.wsattn_prepare(plan, qd, kd)
    fw.wsattn_plan_set_bound(plan, fw.BOUND_WINDOW)
    with pytest.raises(fw.WsattnError) as e:
        fw.wsattn_forward(plan, qd, kd, vd)
    assert e.value.code == 4  # NOT_PREPARED: the statistics depend on the mode
    with pytest.raises(fw.WsattnError) as e:
        fw.wsattn_plan_set_bound(plan, 2)
    assert e.value.code == 1
