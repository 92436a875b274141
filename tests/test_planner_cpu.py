"""The split-KV planner's search on the host: the schedule it returns is the
best of all the chunk sizes it may consider, under its cost model, although
it stops evaluating candidates early.

Cost model (in units of one 96-token tile): every work item costs its tiles
plus 2.5; a plan that splits any request adds 3 (the combine launch) plus, per
split item, the fp32 partial's write and read spread over the CTA pairs.
Candidates split every request into chunks of ceil(max_tiles / k) tiles,
k = 1, 2, ...; each is scored by a longest-processing-time assignment.
"""
import heapq

import numpy as np
import pytest

from test_abi_cpu import TILE, check_schedule

ITEM_OVERHEAD = 2.5
COMBINE_LAUNCH = 3.0


def split_penalty(H):
    return 2.0 * (H * 512 * 4 + H * 4) / (TILE * 576 * 2)


def pieces_for(tiles, chunk):
    out = []
    for b, t in enumerate(tiles):
        if t == 0:
            out.append((b, 0))
            continue
        n = max(1, min((t + chunk - 1) // chunk, t))
        q, r = divmod(t, n)
        out += [(b, q + (1 if i < r else 0)) for i in range(n)]
    return out


def lpt_makespan(costs, nc):
    heap = [(0.0, c) for c in range(nc)]
    heapq.heapify(heap)
    for cost in sorted(costs, reverse=True):
        load, c = heapq.heappop(heap)
        heapq.heappush(heap, (load + cost, c))
    return max(load for load, _ in heap)


def model_cost(pieces, H, nc):
    count = {}
    for b, _ in pieces:
        count[b] = count.get(b, 0) + 1
    costs = [t + ITEM_OVERHEAD for _, t in pieces]
    split_items = sum(1 for b, _ in pieces if count[b] > 1)
    m = lpt_makespan(costs, nc)
    if split_items:
        m += COMBINE_LAUNCH + split_items * split_penalty(H) / nc
    return m


def plan_cost(plan, H, nc):
    """Modelled cost of the schedule the library returned (its own assignment)."""
    load = np.zeros(nc)
    per_request = {}
    items = plan.work_items()
    for (b, t0, t1, slot, cl) in items:
        per_request[b] = per_request.get(b, 0) + 1
    for (b, t0, t1, slot, cl) in items:
        load[cl] += (t1 - t0 + TILE - 1) // TILE + ITEM_OVERHEAD
    split_items = sum(1 for (b, *_rest) in items if per_request[b] > 1)
    m = load.max()
    if split_items:
        m += COMBINE_LAUNCH + split_items * split_penalty(H) / nc
    return m


@pytest.fixture(scope="module")
def m():
    from paged_mla_decode_05_gb300 import build
    build.build()
    import paged_mla_decode_05_gb300 as mod
    return mod


@pytest.mark.parametrize("seed", range(16))
def test_search_returns_the_best_candidate(m, seed):
    rng = np.random.default_rng(100 + seed)
    B = int(rng.choice([1, 3, 8, 40, 200, 600]))
    H = int(rng.choice([16, 64, 128]))
    nc = int(rng.choice([8, 38, 76]))
    long_tail = rng.random() < 0.5
    hi = 40000 if long_tail else 3000
    lens = rng.integers(0, hi, size=B).astype(np.int32)
    max_blocks = int(np.ceil(max(int(lens.max()), 1) / 64)) + 1
    plan = m.mla_decode_plan(B, H, lens, 64, max_blocks, num_clusters=nc, host_only=True)
    tiles = [(int(L) + TILE - 1) // TILE for L in lens]
    max_tiles = max(tiles)
    best = None
    last = -1
    for k in range(1, 257):
        chunk = max(1, (max_tiles + k - 1) // k)
        if chunk == last:
            continue
        last = chunk
        pieces = pieces_for(tiles, chunk)
        if len(pieces) > max(64 * nc, B):
            break
        c = model_cost(pieces, H, nc)
        best = c if best is None else min(best, c)
        if chunk == 1 or max_tiles <= 1:
            break
    got = plan_cost(plan, H, nc)
    assert got <= best + 1e-6, (got, best)
    check_schedule(plan, lens, H, nc)


def test_exchange_pass_fixes_a_known_lpt_miss(m):
    """Two CTA pairs and requests of 3, 3, 2, 2 and 2 tiles (costs 5.5, 5.5,
    4.5, 4.5, 4.5 with the 2.5-tile item overhead). LPT alone ends at 14.5
    ({5.5, 4.5, 4.5} against {5.5, 4.5}). The best split of the five whole
    requests is {5.5, 5.5} against {4.5, 4.5, 4.5}, makespan 13.5: every other
    split leaves one pair at 14.5 or more, and splitting a request costs more
    than it saves here."""
    lens = np.array([3 * TILE, 3 * TILE, 2 * TILE, 2 * TILE, 2 * TILE], dtype=np.int32)
    plan = m.mla_decode_plan(5, 16, lens, 64, 5, num_clusters=2, host_only=True)
    assert all(plan.num_splits(b) == 1 for b in range(5))
    assert plan_cost(plan, 16, 2) == pytest.approx(13.5)
    assert lpt_makespan([5.5, 5.5, 4.5, 4.5, 4.5], 2) == pytest.approx(14.5)
