"""The C-ABI library on a machine without a GPU: it builds, loads, exports
every declared symbol, and its host-only planner produces a valid schedule."""
import ctypes
import subprocess

import numpy as np
import pytest

import mla_workloads as wl

TILE = 96   # tokens per KV tile: work items cover whole tiles


@pytest.fixture(scope="module")
def m():
    from paged_mla_decode_05_gb300 import build
    build.build()
    import paged_mla_decode_05_gb300 as mod
    return mod


def test_exports_every_declared_function(m):
    from paged_mla_decode_05_gb300 import build
    names = m.header_functions()
    assert "mla_decode" in names and "mla_decode_plan" in names
    nm = subprocess.run(["nm", "-D", "--defined-only", build.LIB_PATH], capture_output=True,
                        text=True, check=True).stdout
    exported = {line.split()[-1] for line in nm.splitlines() if " T " in line}
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    lib = ctypes.CDLL(build.LIB_PATH)
    for n in names:
        getattr(lib, n)


def test_status_strings(m):
    assert m.mla_status_string(0) == "ok"
    assert "workspace" in m.mla_status_string(3)


def check_schedule(plan, lens, H, n_clusters):
    """Every (request, head group) is covered exactly once by contiguous
    whole-tile chunks; split chunks own partial slots (shared by the head
    groups of one chunk); the workspace holds them."""
    items = plan.work_items()
    heads = plan.work_item_heads()
    B = len(lens)
    groups = [(g, min(H, g + 128)) for g in range(0, H, 128)]
    covered = {(b, hg): [] for b in range(B) for hg in groups}
    slots = set()
    for (b, t0, t1, slot, cl), hg in zip(items, heads):
        assert 0 <= cl < n_clusters
        assert hg in groups
        assert t0 % TILE == 0 and t0 <= t1 <= lens[b]
        covered[(b, hg)].append((t0, t1, slot))
        if slot >= 0:
            slots.add(slot)
    for (b, hg), segs in covered.items():
        segs = sorted(segs)
        assert len(segs) == plan.num_splits(b)
        if lens[b] == 0:
            assert segs == [(0, 0, -1)]
            continue
        assert segs[0][0] == 0 and segs[-1][1] == lens[b]
        for (a0, a1, _), (b0, _, _) in zip(segs[:-1], segs[1:]):
            assert a1 == b0 and a1 > a0
        if len(segs) == 1:
            assert segs[0][2] == -1
        else:
            assert all(sg[2] >= 0 for sg in segs)
    # the head groups of one chunk share its slot
    by_chunk = {}
    for (b, t0, t1, slot, cl) in items:
        by_chunk.setdefault((b, t0, t1), set()).add(slot)
    assert all(len(v) == 1 for v in by_chunk.values())
    assert sorted(slots) == list(range(len(slots)))
    expect_ws = 0
    if slots:
        o = len(slots) * H * 512 * 4
        o = (o + 255) // 256 * 256
        expect_ws = (o + len(slots) * H * 4 + 255) // 256 * 256
    assert plan.workspace_bytes == expect_ws


@pytest.mark.parametrize("idx", range(5))
def test_schedules_of_the_five_workloads(m, idx):
    spec = wl.WORKLOADS[idx]
    rng = np.random.Generator(np.random.PCG64(spec.seed))
    lens = spec.seq_lens(rng)
    max_blocks = int(np.ceil(spec.max_len / spec.block_size))
    plan = m.mla_decode_plan(spec.B, spec.H, lens, spec.block_size, max_blocks,
                             num_clusters=76, host_only=True)
    check_schedule(plan, lens, spec.H, 76)
    if idx == 3:          # B=512 >> pairs: no split is worth its partial traffic
        assert plan.workspace_bytes == 0
    if idx == 4:          # one 64K request: split across the pairs
        assert plan.num_splits(0) >= 16


@pytest.mark.parametrize("force", [1, 2, 5])
def test_forced_splits(m, force):
    lens = np.array([1000, 96, 0, 97, 5000], dtype=np.int32)
    plan = m.mla_decode_plan(5, 32, lens, 32, 200, num_clusters=8, force_splits=force,
                             host_only=True)
    check_schedule(plan, lens, 32, 8)
    tiles = (lens + TILE - 1) // TILE
    for b in range(5):
        assert plan.num_splits(b) == max(1, min(force, int(tiles[b])))


@pytest.mark.parametrize("H", [129, 256, 300, 1024])
def test_head_groups_cover_every_head(m, H):
    """H > 128: each chunk of each request is scheduled once per group of 128
    heads (the last group holds the rest)."""
    lens = np.array([5000, 96, 0, 1, 3000], dtype=np.int32)
    plan = m.mla_decode_plan(5, H, lens, 32, 200, num_clusters=16, host_only=True)
    check_schedule(plan, lens, H, 16)
    ng = (H + 127) // 128
    assert plan.num_work_items == ng * sum(plan.num_splits(b) for b in range(5))
    forced = m.mla_decode_plan(5, H, lens, 32, 200, num_clusters=16, force_splits=3,
                               host_only=True)
    check_schedule(forced, lens, H, 16)


def test_balance_with_few_pairs(m):
    rng = np.random.default_rng(0)
    lens = rng.integers(1, 4097, size=300).astype(np.int32)
    plan = m.mla_decode_plan(300, 16, lens, 64, 64, num_clusters=10, host_only=True)
    check_schedule(plan, lens, 16, 10)
    load = np.zeros(10)
    for (b, t0, t1, slot, cl) in plan.work_items():
        load[cl] += (t1 - t0 + TILE - 1) // TILE + 2.5
    assert load.max() <= 1.1 * load.mean()


@pytest.mark.parametrize("bad", [dict(B=0), dict(H=0), dict(H=1025), dict(bs=24), dict(bs=256),
                                 dict(len=-1), dict(len=10**5)])
def test_plan_rejects_bad_arguments(m, bad):
    B = bad.get("B", 2)
    lens = np.full(max(B, 1), bad.get("len", 10), dtype=np.int32)[:B] if B else np.zeros(0, np.int32)
    with pytest.raises((m.MLAError, ValueError)):
        m.mla_decode_plan(B, bad.get("H", 8), lens, bad.get("bs", 32), 100, num_clusters=4,
                          host_only=True)


def test_host_only_plan_cannot_decode(m):
    plan = m.mla_decode_plan(1, 8, np.array([10]), 32, 1, num_clusters=2, host_only=True)
    rc = m._lib.LIB.mla_decode(plan.handle, *([ctypes.c_void_p(16)] * 3), 1,
                               *([ctypes.c_void_p(16)] * 2), ctypes.c_float(0.1),
                               *([ctypes.c_void_p(16)] * 3), 0, None)
    assert rc == 1


def test_selftest_argument_checks(m):
    """mla_selftest_wait_timeout rejects a NULL result pointer before touching
    CUDA, and on a machine without a GPU answers 'unsupported device'."""
    lib = m._lib.LIB
    assert lib.mla_selftest_wait_timeout(None, None) == 1          # MLA_ERR_INVALID_ARG
    import torch
    if torch.cuda.is_available():
        pytest.skip("the unsupported-device answer needs a machine without a GPU")
    bits = ctypes.c_uint32(7)
    assert lib.mla_selftest_wait_timeout(None, ctypes.byref(bits)) == 2   # UNSUPPORTED_DEVICE
    assert bits.value == 0


@pytest.mark.parametrize("q_len,H", [(2, 16), (4, 16), (2, 128), (3, 100)])
def test_multi_token_schedule(m, q_len, H):
    """Several query tokens per request: the schedule covers the q_len * H
    query rows of every request (in head groups of 128 rows)."""
    lens = np.array([q_len, 700, 0, 2000, 97], dtype=np.int32)
    plan = m.mla_decode_plan(5, H, lens, 32, 100, num_clusters=16, host_only=True, q_len=q_len)
    check_schedule(plan, lens, q_len * H, 16)
    assert plan.q_shape(512) == (5, q_len, H, 512)


def test_multi_token_argument_checks(m):
    with pytest.raises(m.MLAError):      # a request shorter than its query tokens
        m.mla_decode_plan(2, 16, np.array([3, 100]), 32, 10, num_clusters=4, host_only=True,
                          q_len=4)
    with pytest.raises(m.MLAError):      # more than 1024 query rows per request
        m.mla_decode_plan(2, 128, np.array([30, 100]), 32, 10, num_clusters=4, host_only=True,
                          q_len=9)


def test_sparse_plan_workspace_and_refusals():
    import paged_mla_decode_05_gb300 as m
    B, H, topk = 5, 128, 300
    plan = m.mla_sparse_plan(B, H, topk, num_clusters=76, host_only=True)
    assert plan.workspace_bytes >= B * topk * 4 + B * 4   # row lists and counts
    # every request is planned for topk entries (the bound), in one head group
    covered = {}
    for b, t0, t1, slot, cl in plan.work_items():
        covered[b] = covered.get(b, 0) + (t1 - t0)
    assert covered == {b: topk for b in range(B)}
    with pytest.raises(m.MLAError):
        plan.update(np.full(B, 10, dtype=np.int32))
    for bad in (0, -1):
        with pytest.raises(m.MLAError):
            m.mla_sparse_plan(B, H, bad, num_clusters=76, host_only=True)
