"""Pre-attention producer through the C ABI vs the fp64 oracle (GPU).

wsattn_produce computes y = (W x_t) / rms_t with fp32 accumulation on the
tensor cores, turns the q and k pairs in fp32 and rounds to bf16.  Let
delta bound the fp32 error of y before rounding (C = 3072 exact bf16
products summed in fp32, one multiply by 1/rms, one rotation: a few times
1e-6 relative to sum |w_c x_c| / rms, below 1e-4 absolute for these inputs).
Round-to-nearest bf16 then adds at most half an ulp, at most 2^-8 of the
value, so every element obeys
    |got - want| <= 2^-8 |want| + 2 delta,    delta = 1e-4,
which the tests assert together with a relative L2 error below 3e-3.

Statistics: the plan's statistics after wsattn_produce are those of
wsattn_prepare on the q, k it wrote (the key mean comes from the producer's
column sums, in another fixed order: relative 1e-5), and the forward that
follows agrees with the forward after wsattn_prepare.  Against the oracle,
the statistics of bf16(oracle q, k) agree to 1e-3 (a bf16 rounding that
the fp32 value takes the other way moves a norm by about 1e-4 relative) and
eligibility bit-exactly.
"""
import numpy as np
import pytest
import torch

import oracle
from _helpers import rel_l2
from workloads import Workload, WORKLOADS, producer_inputs, sample_rows

pytestmark = pytest.mark.gpu

EPS = 1e-6
DELTA = 1e-4


def _plan(wl):
    import frame_aligned_window_gb300 as fw
    return fw.wsattn_plan(wl.frames, wl.tokens_per_frame, wl.window, wl.ref_frames, wl.heads,
                          wl.head_dim)


def _produce(wl, model_dim=0):
    import frame_aligned_window_gb300 as fw
    x, w, c, s = producer_inputs(wl, model_dim)
    plan = _plan(wl)
    q, k, v = fw.wsattn_produce(plan, x.cuda(), w.cuda(), c.cuda(), s.cuda(), EPS)
    torch.cuda.synchronize()
    assert fw.wsattn_device_status(plan) == 0
    return plan, (x, w, c, s), (q, k, v)


def _check(got, want):
    g = got.float().cpu().double().numpy()
    err = np.abs(g - want)
    lim = 2.0 ** -8 * np.abs(want) + 2 * DELTA
    assert (err <= lim).all(), float((err - lim).max())
    assert rel_l2(g, want) <= 3e-3


CASES = [
    # name, batch, heads, head_dim, frames, ref, T, grid_w, model_dim
    ("d128_two_tiles_ragged", 2, 2, 128, 2, 1, 80, 8, 256),   # N=240: BN=256, tail of 112 rows
    ("d64_bn128", 1, 2, 64, 4, 1, 48, 8, 192),                # H*D=128: BN=128
    ("d128_bn128", 1, 3, 128, 2, 1, 64, 8, 128),              # H*D=384: BN=128
    ("d64_bn256_four_heads", 2, 4, 64, 3, 1, 48, 8, 320),     # four heads per tile, N=192
    ("short_single_tile", 1, 2, 128, 2, 1, 16, 4, 64),        # N=48 < 128, one k-step
    ("odd_tile_count_batch2", 2, 2, 128, 5, 1, 48, 8, 192),   # N=288: 3 token tiles, the
                                                              # pair's second CTA idles on the last
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_produce_full_parity(case):
    name, B, H, D, F, R, T, gw, C = case
    wl = Workload(name, B, H, D, F, R, T, 1, 40 + len(name), grid_w=gw)
    plan, (x, w, c, s), outs = _produce(wl, C)
    want = oracle.produce(x, w, c, s, EPS, H, D)
    for got, ref in zip(outs, want):
        _check(got, ref)


def test_produce_statistics_match_prepare_and_oracle():
    import frame_aligned_window_gb300 as fw
    wl = Workload("stats", 2, 2, 128, 3, 1, 80, 1, 77, grid_w=8)
    plan, (x, w, c, s), (q, k, v) = _produce(wl, 256)
    st = fw.wsattn_get_stats(plan, wl.batch)
    out_p = fw.wsattn_forward(plan, q, k, v)
    # the same tensors through wsattn_prepare
    plan2 = _plan(wl)
    fw.wsattn_prepare(plan2, q, k)
    st2 = fw.wsattn_get_stats(plan2, wl.batch)
    out2 = fw.wsattn_forward(plan2, q, k, v)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(st["elig"], st2["elig"])
    for key in ("mu", "kmax", "b", "m", "bmax"):
        np.testing.assert_allclose(st[key], st2[key], rtol=1e-5, atol=1e-6)
    # The two row maxima m_i differ by fp32 rounding only (the key mean is
    # summed in another order), but P = bf16(2^(s - m)) can round the other
    # way: each P_ij then moves by at most 2^-8 of itself, and out_i (a
    # P-weighted mean of the v_j, P and l from the same P) by at most
    # 2 * 2^-8 * max |v_j|.  Such flips are rare, so the relative L2
    # difference stays far smaller.
    a, b2 = out_p.cpu().double().numpy(), out2.cpu().double().numpy()
    assert np.abs(a - b2).max() <= 2.0 ** -7 * float(v.float().abs().max())
    assert rel_l2(a, b2) <= 1e-4
    # against the oracle's statistics of its own outputs rounded to bf16
    qo, ko, _ = oracle.produce(x, w, c, s, EPS, wl.heads, wl.head_dim)
    qb = torch.from_numpy(qo).to(torch.bfloat16)
    kb = torch.from_numpy(ko).to(torch.bfloat16)
    want = oracle.prepare(qb, kb, wl.scale)
    assert (np.abs(want["bmax"] - oracle.TAU) / oracle.TAU > 1e-2).all()
    np.testing.assert_array_equal(st["elig"], want["elig"])
    np.testing.assert_allclose(st["mu"], want["mu"], rtol=1e-3, atol=1e-4)
    np.testing.assert_allclose(st["kmax"], want["kmax"], rtol=1e-3)
    np.testing.assert_allclose(st["b"], want["b"].reshape(st["b"].shape), rtol=1e-3)


def test_produce_sr_full_size_sampled():
    # the SR shape (B=1, H=24, D=128, N=22880, C=3072): sampled tokens of
    # every head against the oracle, statistics against wsattn_prepare
    import frame_aligned_window_gb300 as fw
    wl = WORKLOADS["sr"]
    plan, (x, w, c, s), (q, k, v) = _produce(wl)
    rows = sample_rows(wl, n_random=128)
    want = oracle.produce(x, w, c, s, EPS, wl.heads, wl.head_dim, rows=rows)
    for got, ref in zip((q, k, v), want):
        _check(got[:, :, rows], ref)
    st = fw.wsattn_get_stats(plan, wl.batch)
    plan2 = _plan(wl)
    fw.wsattn_prepare(plan2, q, k)
    st2 = fw.wsattn_get_stats(plan2, wl.batch)
    np.testing.assert_array_equal(st["elig"], st2["elig"])
    for key in ("mu", "kmax", "b", "m", "bmax"):
        np.testing.assert_allclose(st[key], st2[key], rtol=1e-5, atol=1e-6)
    # the forward runs on the produced tensors with the folded statistics
    out = fw.wsattn_forward(plan, q, k, v)
    torch.cuda.synchronize()
    assert fw.wsattn_device_status(plan) == 0
    assert torch.isfinite(out).all()


def test_produce_argument_errors():
    import frame_aligned_window_gb300 as fw
    wl = Workload("err", 1, 2, 128, 2, 1, 16, 1, 5)
    x, w, c, s = producer_inputs(wl, 64)
    plan = _plan(wl)
    xd, wd, cd, sd = x.cuda(), w.cuda(), c.cuda(), s.cuda()
    # model_dim not a multiple of 64
    x2 = torch.zeros((1, wl.n_tokens, 96), dtype=torch.bfloat16, device="cuda")
    w2 = torch.zeros((3 * 256, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fw.WsattnError) as e:
        fw.wsattn_produce(plan, x2, w2, cd, sd)
    assert e.value.code == 1
    with pytest.raises(fw.WsattnError) as e:
        fw.wsattn_produce(plan, xd, wd, cd, sd, eps=-1.0)
    assert e.value.code == 1
    # H * D = 64 is not a multiple of 128
    wl1 = Workload("err1", 1, 1, 64, 2, 1, 16, 1, 6)
    x1, w1, c1, s1 = producer_inputs(wl1, 64)
    with pytest.raises(fw.WsattnError) as e:
        fw.wsattn_produce(_plan(wl1), x1.cuda(), w1.cuda(), c1.cuda(), s1.cuda())
    assert e.value.code == 3


@pytest.mark.parametrize("flags", [0, 1])
def test_produce_window_bound_statistics(flags):
    # with window row bounds (and a causal variant) the folded statistics
    # still equal wsattn_prepare's on the same tensors
    import frame_aligned_window_gb300 as fw
    wl = Workload("win", 2, 2, 128, 6, 1, 48, 1, 91 + flags, grid_w=8)
    x, w, c, s = producer_inputs(wl, 128)
    plans = []
    for _ in range(2):
        pl = fw.wsattn_plan(wl.frames, wl.tokens_per_frame, wl.window, wl.ref_frames, wl.heads,
                            wl.head_dim, 0, 0, flags)
        fw.wsattn_plan_set_bound(pl, fw.BOUND_WINDOW)
        plans.append(pl)
    q, k, v = fw.wsattn_produce(plans[0], x.cuda(), w.cuda(), c.cuda(), s.cuda(), EPS)
    fw.wsattn_prepare(plans[1], q, k)
    st, st2 = (fw.wsattn_get_stats(pl, wl.batch) for pl in plans)
    assert fw.wsattn_device_status(plans[0]) == 0
    np.testing.assert_array_equal(st["elig"], st2["elig"])
    for key in ("mu", "kmax", "b", "m", "bmax"):
        np.testing.assert_allclose(st[key], st2[key], rtol=1e-5, atol=1e-6)
