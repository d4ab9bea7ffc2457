"""Benchmark of the frame-aligned window-sparse attention hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl wsattn|reference]
                    [--workload sr] [--block-k 0] [--no-cpu-baseline] [--produce-steps 20]

A step is one pass of the whole hot path over one batch of synthetic input:
wsattn_prepare (key mean, row norms, bounds, eligibility) + wsattn_forward (fused
tcgen05 attention) through the C ABI, on inputs already resident in HBM.  The
plan (block map) is built once per shape, outside the timed region.

Metric: effective TFLOP/s on active blocks = 4 * D * (active query-key pairs)
* B * H per step / step time.  Inputs (q, k, v 140 MB each, out 281 MB at the
SR shape) are larger than L2, so no flush runs between steps.

After the timed steps, `--produce-steps` calls of wsattn_produce (the
pre-attention producer: RMS scale, QKV projection, rotary turn, head packing
and the statistics) are timed on their own and reported under "produce",
against the bf16 tensor peak (2 * B * N * C * 3HD FLOP per call, C = H * D).

Under torchrun every rank runs its own replica of the workload (the path has
no exchange step); value = work of all ranks / the slowest rank's time.
`--impl reference` times the CPU oracle (the reference arm of this build) on
a bounded row sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "effective TFLOP/s on active blocks & % of GB300 bf16 peak; ms/call at SR shape"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}

# dram__bytes_read.sum + dram__bytes_write.sum of one forward launch, from an
# ncu capture, keyed by workload; valid only for the kernel source it was
# measured on (sha256 of forward.cu, first 16 hex digits).
FORWARD_TRAFFIC = {
    ("sr", 80, "4cec5456289a3107"): 1.4867e9,
}


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS, source="fallback")


def _forward_src_hash():
    with open(os.path.join(ROOT, "frame_aligned_window_gb300", "csrc", "forward.cu"), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t_start = self.t_stop = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.reader = threading.Thread(target=self._read, daemon=True)
        self.reader.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark_start(self):
        self.t_start = time.time()

    def mark_stop(self):
        self.t_stop = time.time()

    def stop(self):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def samples_between(self, t0, t1):
        """SM MHz of the samples taken between host times t0 and t1."""
        out = []
        for t, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 2 and t0 <= t <= t1:
                try:
                    out.append(float(parts[1]))
                except ValueError:
                    pass
        return out

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for t, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((t, parts))
        inside = [r for t, r in rows if self.t_start and self.t_stop
                  and self.t_start - 0.2 <= t <= self.t_stop + 0.2]
        use = inside or [r for _, r in rows]
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in use if num(r[1]) is not None]
        mx = [num(r[2]) for r in use if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i in range(4) if r[5 + i] == "Active"})
        pw = [num(r[3]) for r in use if num(r[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "reasons": reasons, "samples": len(use),
                "samples_in_timed_region": len(inside)}


def _dist():
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not dist.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    """Largest value of x across ranks (the job's time is its slowest rank's)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ex2.approx issue rate of one SM, per clock (a probe of this build measured
# 62 G/s per SM at about 1.94 GHz: 32 per clock).
EX2_PER_CLK_PER_SM = 32


def _sfu_line(wl, active_pairs: int, ms: float, clocks):
    """The forward's exponentials per second against the SFU rate at the
    sampled median SM clock (max clock if none was sampled)."""
    import torch
    n = float(active_pairs) * wl.batch * wl.heads
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    summ = clocks.summary() if clocks else {}
    mhz = summ.get("sm_mhz") or summ.get("sm_max_mhz") or 2070.0
    peak = EX2_PER_CLK_PER_SM * sms * mhz * 1e6
    got = n / (ms * 1e-3)
    return {"ex2_per_call": n, "achieved_g_per_s": got / 1e9, "peak_g_per_s": peak / 1e9,
            "frac": got / peak, "peak_source": "probe-measured 32 ex2 per clock per SM x SMs "
                                               "x median SM clock"}


def step_flops(wl, active_pairs: int) -> float:
    return 4.0 * wl.head_dim * active_pairs * wl.batch * wl.heads


# --------------------------------------------------------------- CPU oracle
def oracle_timing(wl, budget_s: float, min_rows: int = 16):
    """Times the oracle on whole heads' rows until `budget_s` is spent.
    Returns (TFLOP/s, seconds, sample description, threads)."""
    import numpy as np
    import oracle
    from workloads import generate

    q, k, v = generate(wl)
    F, T, w, R = wl.frames, wl.tokens_per_frame, wl.window, wl.ref_frames
    n = wl.n_tokens
    m_frames = oracle.blockmap(F, 1, w, R, 1, 1)
    row_pairs = np.zeros(n, dtype=np.int64)  # active keys per query row
    bm = m_frames["bitmap"]
    for a in range(F + R):
        row_pairs[a * T:(a + 1) * T] = int(bm[a].sum()) * T
    qf = q.reshape(-1, n, wl.head_dim)
    kf = k.reshape(-1, n, wl.head_dim)
    vf = v.reshape(-1, n, wl.head_dim)
    flops = 0.0
    rows_done = 0
    heads_done = 0
    t_total = 0.0
    chunk = 2048
    h = 0
    while True:
        qs, ks, vs = qf[h:h + 1], kf[h:h + 1], vf[h:h + 1]
        for r0 in range(0, n, chunk):
            rows = list(range(r0, min(n, r0 + chunk)))
            t0 = time.perf_counter()
            oracle.attention_rows(qs, ks, vs, F, T, w, R, wl.scale, [(0, r) for r in rows])
            t_total += time.perf_counter() - t0
            flops += 4.0 * wl.head_dim * float(row_pairs[rows].sum())
            rows_done += len(rows)
            if t_total >= budget_s and rows_done >= min_rows:
                break
        if rows_done == (h + 1) * n:
            heads_done += 1
        h += 1
        if t_total >= budget_s or h >= qf.shape[0]:
            break
    sample = (f"{rows_done} query rows ({heads_done} whole heads) of {wl.label()}, "
              f"rows in token order, each against every active key")
    return flops / t_total / 1e12, t_total, sample, oracle.num_threads()


def run_reference(args, wl, world, rank):
    """The reference arm: the CPU oracle, on rank 0 only."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    per_step = max(0.05, min(2.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_timing(wl, per_step * 0.2, min_rows=16)
    vals = []
    secs = 0.0
    sample = ""
    threads = 1
    for _ in range(args.steps):
        v, s, sample, threads = oracle_timing(wl, per_step, min_rows=16)
        vals.append(v)
        secs += s
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / max(1, args.steps) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.label(), "block_k": None,
                   "l2": "CPU run; no GPU caches involved"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"per step: {sample}"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm
def run_gpu(args, wl, world, rank, local):
    import torch

    import frame_aligned_window_gb300 as fw
    from workloads import generate

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    q, k, v = generate(wl)
    q_h, k_h, v_h = (x.pin_memory() for x in (q, k, v))
    qd, kd, vd = (x.to(dev) for x in (q, k, v))
    out = torch.empty(q.shape, dtype=torch.float32, device=dev)
    out_h = torch.empty(q.shape, dtype=torch.float32).pin_memory()
    plan = fw.wsattn_plan(wl.frames, wl.tokens_per_frame, wl.window, wl.ref_frames, wl.heads,
                          wl.head_dim, 0, args.block_k)
    flops = step_flops(wl, plan.active_pairs)
    stream = torch.cuda.current_stream()

    def step():
        fw.wsattn_prepare(plan, qd, kd)
        fw.wsattn_forward(plan, qd, kd, vd, out)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    assert fw.wsattn_device_status(plan) == 0

    clocks = ClockSampler(local) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.6)  # let the sampler start before the timed region
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    _barrier(world)
    torch.cuda.synchronize()
    if clocks:
        clocks.mark_start()
    host_t0 = time.time()
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_begin.record(stream)
    for i in range(args.steps):
        e0, e1, e2 = ev[i]
        e0.record(stream)
        fw.wsattn_prepare(plan, qd, kd)
        e1.record(stream)
        fw.wsattn_forward(plan, qd, kd, vd, out)
        e2.record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    _barrier(world)
    if clocks:
        clocks.mark_stop()
    status = fw.wsattn_device_status(plan)
    if status != 0:
        raise RuntimeError(f"device status: {fw.wsattn_status_string(status)}")
    total_ms = t_begin.elapsed_time(t_end)
    prep_ms = [e0.elapsed_time(e1) for e0, e1, _ in ev]
    fwd_ms = [e1.elapsed_time(e2) for _, e1, e2 in ev]
    # The timed steps in (up to) five consecutive bins: forward ms per bin and
    # the SM clock samples that fall inside it (GPU time mapped to host time
    # from the synchronised start), so a drift in time per step can be told
    # apart from a drift in clock.
    bins = []
    nb = min(5, args.steps)
    for i in range(nb):
        a, b = i * args.steps // nb, (i + 1) * args.steps // nb
        if b <= a:
            continue
        t0 = host_t0 + t_begin.elapsed_time(ev[a][0]) * 1e-3
        t1 = host_t0 + t_begin.elapsed_time(ev[b - 1][2]) * 1e-3
        mhz = clocks.samples_between(t0 - 0.1, t1 + 0.1) if clocks else []
        f = statistics.mean(fwd_ms[a:b])
        med = statistics.median(mhz) if mhz else None
        bins.append({"steps": [a, b], "forward_ms": f, "sm_mhz_median": med, "clock_samples": len(mhz),
                     "forward_ms_x_mhz": f * med if med else None})
    ms_step = max_over_ranks(total_ms / args.steps, world)
    # The clock sampler covers the timed steps only: nvidia-smi's queries
    # stall host <-> device copies (the end-to-end loop below ran at 7.2 ms
    # per step beside it, 2.6 ms without).
    if clocks:
        clocks.stop()

    # End to end through the public API: every step copies its inputs in from
    # pinned host memory and its result out to pinned host memory.  Two sets
    # of device buffers let the copies of one step run on their own streams
    # beside the compute of the next (inputs of step i+1 in, result of step
    # i-1 out), as a streaming caller would run it.
    e2e_steps = max(3, min(args.steps, 50))
    q2, k2, v2 = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    out2 = torch.empty_like(out)
    slots = [(qd, kd, vd, out), (q2, k2, v2, out2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    # copies in, compute and copies out each on a stream of their own,
    # ordered by events only
    s_comp = torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of the slot landed
    ev_done = [torch.cuda.Event() for _ in range(2)]  # compute of the slot finished
    ev_out = [torch.cuda.Event() for _ in range(2)]   # result of the slot copied out

    def e2e_run(n_steps, e_begin, e_end):
        s_comp.wait_event(e_begin)
        s_in.wait_event(e_begin)
        for i in range(n_steps):
            sl = i % 2
            qs, ks, vs, os_ = slots[sl]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_done[sl])
                qs.copy_(q_h, non_blocking=True)
                ks.copy_(k_h, non_blocking=True)
                vs.copy_(v_h, non_blocking=True)
                ev_in[sl].record(s_in)
            s_comp.wait_event(ev_in[sl])
            if i >= 2:
                s_comp.wait_event(ev_out[sl])
            with torch.cuda.stream(s_comp):
                fw.wsattn_prepare(plan, qs, ks)
                fw.wsattn_forward(plan, qs, ks, vs, os_)
            ev_done[sl].record(s_comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[sl])
                out_h.copy_(os_, non_blocking=True)
                ev_out[sl].record(s_out)
        for sl in range(2):
            s_comp.wait_event(ev_out[sl])
        e_end.record(s_comp)

    # untimed warm-up: the first transfers from freshly pinned host memory
    # are slow (tens of ms over the first steps), so at least 10 steps
    # whatever --warmup says (with 3, a 20-step run measured 3.7 ms per step
    # against 2.4 once past them)
    w0, w1 = torch.cuda.Event(), torch.cuda.Event()
    w0.record(s_comp)
    e2e_run(max(10, args.warmup), w0, w1)
    torch.cuda.synchronize()
    e_begin = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    _barrier(world)
    torch.cuda.synchronize()
    e_begin.record(s_comp)
    e2e_run(e2e_steps, e_begin, e_end)
    torch.cuda.synchronize()
    _barrier(world)
    e2e_ms = max_over_ranks(e_begin.elapsed_time(e_end) / e2e_steps, world)

    # The pre-attention producer (x -> q, k, v plus the statistics), timed on
    # its own: one wsattn_produce call per iteration, inputs resident in HBM.
    prod = None
    if args.produce_steps > 0 and (wl.heads * wl.head_dim) % 128 == 0:
        from workloads import producer_inputs
        x, w, rc_, rs_ = (t.to(dev) for t in producer_inputs(wl))
        pq, pk, pv = (torch.empty_like(qd) for _ in range(3))
        for _ in range(3):
            fw.wsattn_produce(plan, x, w, rc_, rs_, 1e-6, pq, pk, pv)
        torch.cuda.synchronize()
        pe = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.produce_steps)]
        for a, b in pe:
            a.record(stream)
            fw.wsattn_produce(plan, x, w, rc_, rs_, 1e-6, pq, pk, pv)
            b.record(stream)
        torch.cuda.synchronize()
        if fw.wsattn_device_status(plan) != 0:
            raise RuntimeError("device status after wsattn_produce")
        p_ms = statistics.mean(a.elapsed_time(b) for a, b in pe)
        C = x.shape[2]
        p_flops = 2.0 * wl.batch * wl.n_tokens * C * 3 * wl.heads * wl.head_dim
        prod = {"ms_per_call": p_ms, "calls": args.produce_steps, "model_dim": C,
                "gflop_per_call": p_flops / 1e9, "launches": 4,
                "includes": "RMS pre-pass, projection GEMM, key-sum reduction and the "
                            "statistics pass",
                "achieved_tflops": p_flops / (p_ms * 1e-3) / 1e12}
        del x, w, rc_, rs_, pq, pk, pv

    if rank != 0:
        return None
    peaks = _peaks()
    fwd_avg = statistics.mean(fwd_ms)
    prep_avg = statistics.mean(prep_ms)
    achieved = flops / (fwd_avg * 1e-3) / 1e12
    elem = q.numel()
    prep_bytes = 3 * elem * 2 + 2 * wl.batch * wl.heads * wl.n_tokens * 4
    src = _forward_src_hash()
    traffic = FORWARD_TRAFFIC.get((wl.name, plan.block_k, src))
    line = {
        "metric": METRIC,
        "value": flops * world / (ms_step * 1e-3) / 1e12,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": wl.label(), "block_q": plan.block_q, "block_k": plan.block_k,
                   "gflop_per_step": flops / 1e9,
                   "l2": "inputs larger than L2 (q, k, v, out = %.0f MB); no flush"
                         % ((3 * elem * 2 + elem * 4) / 1e6),
                   "per_rank": "independent replica"},
        "roofline": {"bound": "tensor", "kernel": "wsattn_fwd_kernel", "achieved": achieved,
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": achieved / peaks["bf16_tflops"], "traffic": traffic,
                     "traffic_unit": "bytes per launch (ncu dram read + write)",
                     "algorithmic_bytes": 3 * elem * 2 + elem * 4,
                     "peak_source": f"{peaks['source']} (bf16 burst)",
                     "ms_per_launch": fwd_avg,
                     "ms_per_launch_median": statistics.median(fwd_ms),
                     # the secondary limit: one ex2 per active (query, key) pair
                     "sfu": _sfu_line(wl, plan.active_pairs, fwd_avg, clocks)},
        "prepare": {"bound": "hbm", "ms_per_call": prep_avg, "launches": 2,
                    "algorithmic_bytes": prep_bytes,
                    "achieved": prep_bytes / (prep_avg * 1e-3) / 1e9,
                    "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": prep_bytes / (prep_avg * 1e-3) / 1e9 / peaks["hbm_gbs"]},
        "e2e": {"value": flops * world / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": 3 * elem * 2,
                "d2h_bytes_per_step": elem * 4,
                "copies": "pinned host <-> device on two copy streams, overlapping the "
                          "compute of the neighbouring steps (double-buffered device side)"},
        "produce": None if prod is None else dict(
            prod, bound="tensor", peak=peaks["bf16_tflops"], unit="TFLOP/s",
            frac=prod["achieved_tflops"] / peaks["bf16_tflops"]),
        "gpu_launches": 3 * args.steps,
        "clocks": clocks.summary() if clocks else None,
        "step_bins": bins,
    }
    return line


def time_config(name, steps, warmup, local, peaks):
    """One other workload: prepare + forward `steps` times on resident inputs,
    CUDA-event times per launch, its own clock record and roofline line."""
    import torch

    import frame_aligned_window_gb300 as fw
    from workloads import WORKLOADS, generate

    wl = WORKLOADS[name]
    dev = torch.device("cuda", local)
    q, k, v = (x.to(dev) for x in generate(wl))
    out = torch.empty(q.shape, dtype=torch.float32, device=dev)
    plan = fw.wsattn_plan(wl.frames, wl.tokens_per_frame, wl.window, wl.ref_frames, wl.heads,
                          wl.head_dim)
    flops = step_flops(wl, plan.active_pairs)
    stream = torch.cuda.current_stream()
    for _ in range(max(3, warmup)):
        fw.wsattn_prepare(plan, q, k)
        fw.wsattn_forward(plan, q, k, v, out)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.6)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    clocks.mark_start()
    for e0, e1, e2 in ev:
        e0.record(stream)
        fw.wsattn_prepare(plan, q, k)
        e1.record(stream)
        fw.wsattn_forward(plan, q, k, v, out)
        e2.record(stream)
    torch.cuda.synchronize()
    clocks.mark_stop()
    clocks.stop()
    status = fw.wsattn_device_status(plan)
    if status != 0:
        raise RuntimeError(f"{name}: device status {fw.wsattn_status_string(status)}")
    fwd = statistics.mean(b.elapsed_time(c) for _, b, c in ev)
    prep = statistics.mean(a.elapsed_time(b) for a, b, _ in ev)
    step = statistics.mean(a.elapsed_time(c) for a, _, c in ev)
    achieved = flops / (fwd * 1e-3) / 1e12
    res = {"workload": wl.label(), "block_k": plan.block_k, "steps": steps,
           "gflop_per_call": flops / 1e9, "ms_per_forward": fwd, "ms_per_prepare": prep,
           "ms_per_step": step,
           "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                        "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                        "peak_source": f"{peaks['source']} (bf16 burst)"},
           "clocks": clocks.summary()}
    if name in ("tiny", "small"):
        res["note"] = "latency-bound: fewer work items than SMs' worth of steps"
    del q, k, v, out
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="wsattn", choices=["wsattn", "reference"])
    ap.add_argument("--workload", default="sr")
    ap.add_argument("--block-k", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--produce-steps", type=int, default=20,
                    help="wsattn_produce calls timed after the attention steps (0: none)")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle time for the cpu_baseline sample")
    ap.add_argument("--other-configs", default="sr_long,dense,small,tiny",
                    help="comma-separated workloads timed after the main one (rank 0, N=1 "
                         "only); 'none' or '' for none")
    args = ap.parse_args()
    from workloads import WORKLOADS
    wl = WORKLOADS[args.workload]
    world, rank, local = _dist()
    if args.impl == "reference":
        run_reference(args, wl, world, rank)
        return
    line = run_gpu(args, wl, world, rank, local)
    if (rank == 0 and line is not None and world == 1 and args.other_configs
            and args.other_configs != "none"):
        steps_of = {"sr_long": 30, "dense": 30, "sr": 60, "small": 200, "tiny": 200}
        line["configs"] = {}
        for name in [x for x in args.other_configs.split(",") if x and x != wl.name]:
            line["configs"][name] = time_config(name, steps_of.get(name, 30), args.warmup, local,
                                                _peaks())
    if rank == 0 and line is not None:
        if not args.no_cpu_baseline and world == 1:
            v, secs, sample, threads = oracle_timing(wl, args.cpu_budget)
            line["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", "cores": threads,
                                    "kind": "oracle", "sample": sample,
                                    "seconds": secs}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
