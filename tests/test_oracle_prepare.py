"""Pins for the oracle's fixed-max statistics (CPU only).

Google Developers Blog post "HeyGen x Google Cloud: Bringing Avatar IV to
TPUs", section "Breaking softmax's dependency chain": keys are mean-centered;
a row's logits are bounded by its query norm times the max key norm
(Cauchy-Schwarz); heads whose bound is too loose are not eligible.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from workloads import WORKLOADS, generate, micro


def test_hand_worked_statistics(golden):
    vals = {ln.split()[0]: [float(x) for x in ln.split()[1:]] for ln in golden("prepare_micro.txt")}
    k = torch.tensor(vals["k"], dtype=torch.float64).reshape(1, 4, 2)
    q = torch.tensor(vals["q"], dtype=torch.float64).reshape(1, 4, 2)
    st = oracle.prepare(q, k, 1.0 / math.sqrt(2.0))
    np.testing.assert_allclose(st["mu"][0], vals["mu"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(st["kmax"], vals["kmax"], rtol=1e-15)
    np.testing.assert_allclose(st["qn"][0], vals["qn"], rtol=1e-15)
    np.testing.assert_allclose(st["b"][0], vals["b"], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(st["bmax"], vals["bmax"], rtol=1e-14)
    assert st["elig"][0] == 1


@pytest.mark.parametrize("seed", [31, 32, 33])
def test_statistics_match_python_loops(seed):
    wl, q, k, v = micro(seed, 1, 2, 8, 3, 1, 5, 1)
    st = oracle.prepare(q, k, wl.scale)
    qf = q.to(torch.float64).reshape(2, wl.n_tokens, 8).tolist()
    kf = k.to(torch.float64).reshape(2, wl.n_tokens, 8).tolist()
    for h in range(2):
        mu = brute.key_mean(kf[h])
        km = max(brute.norm([a - b for a, b in zip(row, mu)]) for row in kf[h])
        np.testing.assert_allclose(st["mu"][h], mu, rtol=1e-13)
        np.testing.assert_allclose(st["kmax"][h], km, rtol=1e-13)
        for i, row in enumerate(qf[h]):
            b = wl.scale * brute.norm(row) * km
            np.testing.assert_allclose(st["b"][h][i], b, rtol=1e-13)
        assert st["bmax"][h] == max(st["b"][h])


def test_centering_tightens_bound():
    # the shared key offset inflates the uncentered bound
    wl = WORKLOADS["tiny"]
    q, k, v = generate(wl)
    st = oracle.prepare(q, k, wl.scale)
    kd = oracle.as_f64(k)
    unc = [np.linalg.norm(kd[h], axis=1).max() for h in range(wl.heads)]
    assert all(st["kmax"][h] < unc[h] for h in range(wl.heads))


def _one_head(bmax_target, d=4):
    """q with one row of norm r, k centered with norm 1 rows -> bmax = scale * r."""
    scale = 1.0 / math.sqrt(d)
    r = bmax_target / scale
    q = torch.zeros(1, 2, d, dtype=torch.float64)
    q[0, 0, 0] = r
    k = torch.zeros(1, 2, d, dtype=torch.float64)
    k[0, 0, 0], k[0, 1, 0] = 1.0, -1.0
    return q, k, scale


def test_eligibility_threshold_and_tie():
    q, k, s = _one_head(40.0)
    st = oracle.prepare(q, k, s, tau=40.0)
    assert st["bmax"][0] == pytest.approx(40.0, rel=1e-15)
    assert st["elig"][0] == (st["bmax"][0] <= 40.0)
    q, k, s = _one_head(40.5)
    assert oracle.prepare(q, k, s, tau=40.0)["elig"][0] == 0
    q, k, s = _one_head(39.5)
    assert oracle.prepare(q, k, s, tau=40.0)["elig"][0] == 1


def test_underflow_clause_binds_above_43_67():
    # with tau raised to 50, a bound of 44 passes tau but 2*44 >= 126 ln 2
    q, k, s = _one_head(44.0)
    assert oracle.prepare(q, k, s, tau=50.0)["elig"][0] == 0
    q, k, s = _one_head(43.0)
    assert oracle.prepare(q, k, s, tau=50.0)["elig"][0] == 1


@pytest.mark.parametrize("name", ["tiny", "small"])
def test_workload_heads_eligible_with_margin(name):
    wl = WORKLOADS[name]
    q, k, v = generate(wl)
    st = oracle.prepare(q, k, wl.scale)
    assert st["elig"].all()
    assert (np.abs(st["bmax"] - oracle.TAU) / oracle.TAU > 1e-3).all()
