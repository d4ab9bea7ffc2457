"""The forward's host-built work schedule (CPU: wsattn_get_schedule runs
the same builder the forward uses, with no GPU).

Every work item is dealt to exactly one CTA, each CTA's list keeps the
kernel's item order (longest class first), and the greedy longest-first
deal keeps the predicted per-CTA work within one item's cost of the mean.
The cost model (1600 cycles per key step + 3500 per tile, in units of 100
cycles) is restated here from the tiles' step counts, which follow from the
frame structure: a run of L consecutive active key blocks takes
ceil(L / G) steps."""
import math

import pytest

import frame_aligned_window_gb300 as fw
from workloads import WORKLOADS


def _item_costs(plan, batch):
    """Per work item (kernel order), the predicted cost, from the frame
    structure: query frame a attends key frames within the window plus the
    reference frames; consecutive attended frames form runs."""
    F, T, w, R = plan.frames, plan.tokens_per_frame, plan.window, plan.ref_frames
    bk = plan.block_k
    G = max(1, 160 // bk)
    bpf = T // bk                        # key blocks per frame
    tiles_per_frame = math.ceil(T / 128)
    per_frame = []
    for a in range(F + R):
        att = [c for c in range(F + R)
               if c < R or a < R or abs((a - R) - (c - R)) <= w]
        runs, start, prev = [], None, None
        for c in att:
            if start is None:
                start = prev = c
            elif c == prev + 1:
                prev = c
            else:
                runs.append(prev - start + 1)
                start = prev = c
        runs.append(prev - start + 1)
        nstep = sum(math.ceil(r * bpf / G) for r in runs)
        nblk = len(att) * bpf
        per_frame.append((nblk, nstep))
    tiles = []
    for a, (nblk, nstep) in enumerate(per_frame):
        tiles += [(nblk, nstep, a)] * tiles_per_frame
    tiles.sort(key=lambda t: -t[0])      # stable: longest class first
    classes = []
    for t in tiles:
        if classes and classes[-1][0][0] == t[0]:
            classes[-1].append(t)
        else:
            classes.append([t])
    BH = batch * plan.heads
    costs = []
    for cl in classes:
        for o in range(len(cl) * BH):
            costs.append(16 * cl[o % len(cl)][1] + 35)
    return costs


@pytest.mark.parametrize("name,batch,grid", [("tiny", 1, 7), ("small", 2, 152),
                                              ("sr", 1, 152), ("dense", 2, 152)])
def test_schedule_is_a_balanced_partition(name, batch, grid):
    wl = WORKLOADS[name]
    plan = fw.wsattn_plan(wl.frames, wl.tokens_per_frame, wl.window, wl.ref_frames, wl.heads,
                          wl.head_dim)
    n_items = plan.tiles_per_head * batch * wl.heads
    grid = min(grid, n_items)
    lists = fw.wsattn_get_schedule(plan, batch, grid)
    flat = [i for lst in lists for i in lst]
    assert sorted(flat) == list(range(n_items))            # each item exactly once
    assert all(lst == sorted(lst) for lst in lists)         # kernel order kept
    costs = _item_costs(plan, batch)
    assert len(costs) == n_items
    loads = [sum(costs[i] for i in lst) for lst in lists]
    mean = sum(costs) / grid
    assert max(loads) <= mean + max(costs)


def test_schedule_beats_round_robin_at_sr():
    wl = WORKLOADS["sr"]
    plan = fw.wsattn_plan(wl.frames, wl.tokens_per_frame, wl.window, wl.ref_frames, wl.heads,
                          wl.head_dim)
    grid = 152
    costs = _item_costs(plan, 1)
    lists = fw.wsattn_get_schedule(plan, 1, grid)
    greedy = max(sum(costs[i] for i in lst) for lst in lists)
    rr = max(sum(costs[i] for i in range(c, len(costs), grid)) for c in range(grid))
    assert greedy < rr
    assert greedy <= 1.02 * sum(costs) / grid


def test_schedule_argument_errors():
    wl = WORKLOADS["tiny"]
    plan = fw.wsattn_plan(wl.frames, wl.tokens_per_frame, wl.window, wl.ref_frames, wl.heads,
                          wl.head_dim)
    for batch, grid in ((0, 4), (1, 0)):
        with pytest.raises(fw.WsattnError) as e:
            fw.wsattn_get_schedule(plan, batch, grid)
        assert e.value.code == 1
