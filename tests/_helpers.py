"""Shared helpers for the parity tests (oracle side and CUDA side)."""
import numpy as np
import torch

import oracle
from workloads import WORKLOADS

# Parity bar for fp32 outputs from bf16 inputs.
TOL_MAX_ABS = 1e-2
TOL_REL_L2 = 5e-3


def rel_l2(got, want) -> float:
    return float(np.linalg.norm(got - want) / np.linalg.norm(want))


def flat_heads(x, wl):
    return x.reshape(-1, wl.n_tokens, wl.head_dim)


def select_heads(x, wl, bh_list):
    """[B, H, N, D] tensor -> [len(bh_list), N, D] for the listed (b, h)."""
    idx = [b * wl.heads + h for b, h in bh_list]
    return flat_heads(x, wl)[idx]


def oracle_rows(wl, q, k, v, bh_list, rows) -> np.ndarray:
    """Oracle output for `rows` of each listed (b, h): [len(bh_list), len(rows), D]."""
    qs, ks, vs = (select_heads(x, wl, bh_list) for x in (q, k, v))
    pairs = [(i, r) for i in range(len(bh_list)) for r in rows]
    out = oracle.attention_rows(qs, ks, vs, wl.frames, wl.tokens_per_frame, wl.window,
                                wl.ref_frames, wl.scale, pairs)
    return out.reshape(len(bh_list), len(rows), wl.head_dim)


def oracle_prepare_all(wl, q, k, chunk=8, tau=oracle.TAU) -> dict:
    """fp64 statistics of every (b, h), computed a few heads at a time."""
    qf, kf = flat_heads(q, wl), flat_heads(k, wl)
    parts = []
    for s in range(0, qf.shape[0], chunk):
        parts.append(oracle.prepare(qf[s:s + chunk], kf[s:s + chunk], wl.scale, tau))
    return {key: np.concatenate([p[key] for p in parts]) for key in parts[0]}


def gpu_run(wl, q, k, v, block_k=0, force_path=-1, tau=0.0, mask_flags=0, bound=0):
    """Plan, prepare and forward through the library; returns (plan, out, k_centered)."""
    import frame_aligned_window_gb300 as fw
    plan = fw.wsattn_plan(wl.frames, wl.tokens_per_frame, wl.window, wl.ref_frames, wl.heads,
                          wl.head_dim, 0, block_k, mask_flags)
    if bound:
        fw.wsattn_plan_set_bound(plan, bound)
    if force_path >= 0 or tau > 0:
        fw.wsattn_plan_set_debug(plan, force_path, tau)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    fw.wsattn_prepare(plan, qd, kd)
    out = fw.wsattn_forward(plan, qd, kd, vd)
    torch.cuda.synchronize()
    st = fw.wsattn_device_status(plan)
    assert st == 0, fw.wsattn_status_string(st)
    return plan, out, kd


def workload(name):
    return WORKLOADS[name]
