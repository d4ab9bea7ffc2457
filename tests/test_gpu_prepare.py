"""Prepare kernel vs the oracle's fp64 statistics (GPU).

Eligibility flags are compared bit-exactly, with the margin |B_h - tau| / tau
> 1e-3 asserted so that fp32-vs-fp64 rounding cannot decide a flag.  The
statistics are fp32 reductions of the exact bf16 inputs, so they agree with
the fp64 oracle to fp32 rounding: relative 1e-5 (absolute 2e-5 for the mean,
whose entries can be near zero).  The row shift m_i = b_i + scale q_i.mu is
checked against the same expression evaluated from the oracle's mean.
"""
import numpy as np
import pytest
import torch

import oracle
from _helpers import flat_heads, oracle_prepare_all, workload
from workloads import generate

pytestmark = pytest.mark.gpu

REL_BOUND = 1e-5


@pytest.mark.parametrize("name", ["tiny", "small", "sr", "sr_long", "dense"])
def test_prepare_matches_oracle(name):
    import frame_aligned_window_gb300 as fw
    wl = workload(name)
    q, k, v = generate(wl)
    plan = fw.wsattn_plan(wl.frames, wl.tokens_per_frame, wl.window, wl.ref_frames, wl.heads,
                          wl.head_dim)
    qd, kd = q.cuda(), k.cuda()
    fw.wsattn_prepare(plan, qd, kd)
    st = fw.wsattn_get_stats(plan, wl.batch)
    assert fw.wsattn_device_status(plan) == 0
    assert torch.equal(kd.cpu(), k) and torch.equal(qd.cpu(), q)  # read only
    want = oracle_prepare_all(wl, q, k)
    # eligibility: bit-exact, away from the threshold
    assert (np.abs(want["bmax"] - oracle.TAU) / oracle.TAU > 1e-3).all()
    np.testing.assert_array_equal(st["elig"], want["elig"])
    np.testing.assert_allclose(st["mu"], want["mu"], rtol=0, atol=2e-5)
    np.testing.assert_allclose(st["kmax"], want["kmax"], rtol=REL_BOUND)
    np.testing.assert_allclose(st["bmax"], want["bmax"], rtol=REL_BOUND)
    np.testing.assert_allclose(st["b"], want["b"], rtol=REL_BOUND, atol=1e-6)
    # B_h is exactly the max of the kernel's own row bounds
    np.testing.assert_array_equal(st["bmax"], st["b"].max(axis=1))
    # row shift: m_i = b_i + scale q_i.mu (the bound on uncentered logits)
    qf = flat_heads(q, wl).double().numpy()
    c = wl.scale * np.einsum("hnd,hd->hn", qf, want["mu"])
    np.testing.assert_allclose(st["m"], want["b"] + c, rtol=0,
                               atol=1e-5 * (1 + np.abs(want["b"] + c).max()))
    if name == "sr_long":
        bad = {b * wl.heads + h for b in range(wl.batch) for h in wl.boost_heads}
        assert {i for i in range(len(st["elig"])) if st["elig"][i] == 0} == bad
    else:
        assert st["elig"].all()


def test_prepare_is_deterministic():
    import frame_aligned_window_gb300 as fw
    wl = workload("small")
    q, k, v = generate(wl)
    plan = fw.wsattn_plan(wl.frames, wl.tokens_per_frame, wl.window, wl.ref_frames, wl.heads,
                          wl.head_dim)
    res = []
    for _ in range(2):
        qd, kd = q.cuda(), k.cuda()
        fw.wsattn_prepare(plan, qd, kd)
        st = fw.wsattn_get_stats(plan, wl.batch)
        res.append((kd.cpu(), st))
    assert torch.equal(res[0][0], res[1][0])
    for key in ("b", "mu", "kmax", "bmax", "elig"):
        np.testing.assert_array_equal(res[0][1][key], res[1][1][key])


def test_tau_override_changes_eligibility():
    import frame_aligned_window_gb300 as fw
    wl = workload("small")
    q, k, v = generate(wl)
    plan = fw.wsattn_plan(wl.frames, wl.tokens_per_frame, wl.window, wl.ref_frames, wl.heads,
                          wl.head_dim)
    fw.wsattn_plan_set_debug(plan, -1, 10.0)  # every head of 'small' has B_h in 16..17
    qd, kd = q.cuda(), k.cuda()
    fw.wsattn_prepare(plan, qd, kd)
    st = fw.wsattn_get_stats(plan, wl.batch)
    want = oracle_prepare_all(wl, q, k, tau=10.0)
    np.testing.assert_array_equal(st["elig"], want["elig"])
    assert not st["elig"].any()


def test_underflow_clause_decides_eligibility_and_forward_matches():
    # Google Developers Blog post "HeyGen x Google Cloud: Bringing Avatar IV
    # to TPUs", section "Breaking softmax's dependency chain": with a loose
    # bound the fixed-max exponentials underflow.  With tau raised to 50, a
    # head whose B_h lies in (63 ln 2, 50] = (43.67, 50] passes the tau test
    # but fails the row clause 2 b_i < 126 ln 2, so it must run the online
    # path.  Head 3 of 'small' gets its queries scaled so that B_h is about 46;
    # the other heads stay near 17.
    import frame_aligned_window_gb300 as fw
    from _helpers import gpu_run, oracle_rows, rel_l2, TOL_MAX_ABS, TOL_REL_L2
    wl = workload("small")
    q, k, v = generate(wl)
    base = oracle_prepare_all(wl, q, k)
    head = 3
    q = q.clone()
    q[0, head] = (q[0, head].double() * (46.0 / base["bmax"][head])).to(torch.bfloat16)
    tau = 50.0
    want = oracle_prepare_all(wl, q, k, tau=tau)
    limit = 63.0 * np.log(2.0)
    assert limit * 1.001 < want["bmax"][head] < tau / 1.001
    assert (np.delete(want["bmax"], head) < limit / 1.001).all()
    assert want["elig"][head] == 0 and np.delete(want["elig"], head).all()
    plan, out, _ = gpu_run(wl, q, k, v, tau=tau)
    st = fw.wsattn_get_stats(plan, wl.batch)
    np.testing.assert_array_equal(st["elig"], want["elig"])
    np.testing.assert_allclose(st["bmax"], want["bmax"], rtol=REL_BOUND)
    # the ineligible head's output (every row) against the oracle
    rows = list(range(wl.n_tokens))
    ref = oracle_rows(wl, q, k, v, [(0, head)], rows)[0]
    got = flat_heads(out.cpu(), wl)[head].double().numpy()
    err = float(np.abs(got - ref).max())
    assert err <= TOL_MAX_ABS and rel_l2(got, ref) <= TOL_REL_L2, err
