"""GPU parity of the sm_103a decode (through the C ABI) against the fp64 oracle.

Every workload, the B=512, H=128 one the benchmark times included, is compared
element by element over every (request, head), in the launch configuration the
benchmark uses (the planner's own choice of pairs and splits).
"""
import numpy as np
import pytest

import mla_workloads as wl
from gpu_helpers import (LSE_ATOL, OUT_ATOL, OUT_RTOL, assert_parity, oracle_args, run_library,
                         spec, to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for -m gpu tests")
    from paged_mla_decode_05_gb300 import build
    build.build()
    import paged_mla_decode_05_gb300 as m
    assert m.mla_device_supported(), "needs an sm_103 device"
    return m


def full_parity(oracle_mod, w, **kw):
    out, lse, plan = run_library(w, **kw)
    ref_out, ref_lse = oracle_mod.mla_decode(*oracle_args(w))
    assert_parity(out, lse, ref_out, ref_lse, w["name"])
    return out, lse, plan


def test_tiny_config(lib, oracle_mod):
    full_parity(oracle_mod, wl.generate(wl.WORKLOADS[0]))


def test_v2lite_config_head_padding(lib, oracle_mod):
    w = wl.generate(wl.WORKLOADS[1])
    _, _, plan = full_parity(oracle_mod, w)
    assert plan.num_work_items >= w["B"]


@pytest.mark.parametrize("idx", [2, 3, 4])
def test_large_configs_full(lib, oracle_mod, idx):
    """R1 B=128, R1 B=512 (the benchmark workload) and the long-context split
    workload, every (request, head) row against the full oracle."""
    w = wl.generate(wl.WORKLOADS[idx])
    _, _, plan = full_parity(oracle_mod, w)
    if idx == 4:   # the 64K request must be split across pairs and recombined
        assert plan.num_splits(0) > 1


def test_output_only_16_byte_aligned(lib, oracle_mod):
    """The epilogue writes 32 bytes per lane where out is 32-byte aligned and
    16 bytes per lane otherwise: an out that starts 16 bytes past a 32-byte
    boundary takes the second path, with the same results (bit for bit) as
    an aligned out, and nothing is written before its first element."""
    import torch
    import paged_mla_decode_05_gb300 as m
    from gpu_helpers import decode_into
    w = spec("a16", 3, 128, 32, [1, 300, 1000], seed=21)
    t = to_device(w)
    B, H = int(w["B"]), int(w["H"])
    plan = m.mla_decode_plan(B, H, w["seq_lens"], int(w["block_size"]), int(w["max_blocks"]))
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device="cuda")
    n = B * H * 512
    buf = torch.full((n + 16,), float("nan"), dtype=torch.bfloat16, device="cuda")
    assert buf.data_ptr() % 32 == 0
    out16 = buf[8:8 + n].view(B, H, 512)          # 16 bytes past a 32-byte boundary
    assert out16.data_ptr() % 32 == 16
    out32 = torch.full((B, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse16 = torch.empty((B, H), dtype=torch.float32, device="cuda")
    lse32 = torch.empty((B, H), dtype=torch.float32, device="cuda")
    decode_into(m, plan, w, t, t["q_nope"], t["q_pe"], out16, lse16, ws)
    decode_into(m, plan, w, t, t["q_nope"], t["q_pe"], out32, lse32, ws)
    assert m.mla_check_device_error(plan) == 0
    assert torch.isnan(buf[:8]).all() and torch.isnan(buf[8 + n:]).all()
    assert torch.equal(out16.view(torch.int16), out32.view(torch.int16))
    assert torch.equal(lse16, lse32)
    ref_out, ref_lse = oracle_mod.mla_decode(*oracle_args(w))
    assert_parity(out16.float().cpu().numpy().astype(np.float64),
                  lse16.cpu().numpy().astype(np.float64), ref_out, ref_lse, "a16")


@pytest.mark.parametrize("H", [1, 7, 32, 100, 128])
def test_head_counts(lib, oracle_mod, H):
    full_parity(oracle_mod, spec(f"h{H}", 3, H, 32, [1, 97, 300], seed=H))


@pytest.mark.parametrize("H,splits", [(129, 0), (192, 2), (256, 0)])
def test_head_groups_above_128(lib, oracle_mod, H, splits):
    """More than 128 query heads: the plan runs each KV chunk once per group of
    128 heads (the last group padded inside the kernel), every row against
    the oracle, with and without split partials."""
    w = spec(f"h{H}", 3, H, 32, [1, 700, 1300], seed=H)
    _, _, plan = full_parity(oracle_mod, w, force_splits=splits)
    heads = plan.work_item_heads()
    assert {h for h, _ in heads} == set(range(0, H, 128))


@pytest.mark.parametrize("bs", [16, 32, 64, 128])
def test_block_sizes_ragged(lib, oracle_mod, bs):
    lens = [1, 15, 95, 96, 97, 191, 192, 193, 500]
    full_parity(oracle_mod, spec(f"bs{bs}", len(lens), 16, bs, lens, seed=bs))


def test_empty_and_tiny_requests(lib, oracle_mod):
    w = spec("empty", 4, 8, 32, [0, 1, 0, 2], seed=3)
    out, lse, _ = full_parity(oracle_mod, w)
    assert np.all(out[0] == 0) and np.all(lse[0] == -np.inf)


def split_partials(w, force_splits):
    """Decode with forced splits and return the plan, its work items and the
    fp32 partials the decode kernel left in the workspace, before the combine.

    Workspace layout (written by the decode kernel, read by the combine): the
    partial outputs fp32 [slots, H, 512] at offset 0, then the partial
    log-sum-exps fp32 [slots, H] at the next 256-byte boundary."""
    import torch
    import paged_mla_decode_05_gb300 as m
    t = to_device(w)
    B, H = int(w["B"]), int(w["H"])
    plan = m.mla_decode_plan(B, H, w["seq_lens"], int(w["block_size"]), int(w["max_blocks"]),
                             force_splits=force_splits)
    out = torch.empty((B, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    m.mla_decode(plan, t["q_nope"], t["q_pe"], t["kv_cache"], t["block_table"], t["seq_lens"],
                 float(w["sm_scale"]), out, lse, ws)
    assert m.mla_check_device_error(plan) == 0
    items = plan.work_items()
    slots = sum(1 for it in items if it[3] >= 0)
    o_bytes = slots * H * 512 * 4
    raw = ws.cpu().numpy()
    part_o = raw[:o_bytes].view(np.float32).reshape(slots, H, 512).astype(np.float64)
    l_off = (o_bytes + 255) // 256 * 256
    part_lse = raw[l_off:l_off + slots * H * 4].view(np.float32).reshape(slots, H).astype(np.float64)
    return plan, items, part_o, part_lse


@pytest.mark.parametrize("splits", [2, 3, 7])
def test_forced_splits_match_oracle(lib, oracle_mod, splits):
    w = spec("split", 3, 128, 64, [1000, 96 * 5 + 1, 50], seed=splits, peaky_fraction=0.02)
    full_parity(oracle_mod, w)
    _, _, plan = full_parity(oracle_mod, w, force_splits=splits)
    assert plan.num_splits(0) == splits and plan.workspace_bytes > 0


@pytest.mark.parametrize("splits", [2, 7])
def test_split_partials_match_oracle_partial(lib, oracle_mod, splits):
    """Each split's fp32 partial (normalised over its own token range) and its
    log-sum-exp, as the decode kernel wrote them before the combine, against
    the oracle's partial of the same range: this checks the partial writer on
    its own, so a fault in it cannot hide behind the combine."""
    w = spec("split", 3, 128, 64, [1000, 96 * 5 + 1, 50], seed=splits, peaky_fraction=0.02)
    plan, items, part_o, part_lse = split_partials(w, splits)
    args = oracle_args(w)
    checked = 0
    for (b, t0, t1, slot, _cluster) in items:
        if slot < 0:
            continue
        for h in range(int(w["H"])):
            ref_o, ref_l = oracle_mod.mla_partial(*args, b, h, t0, t1)
            err = np.abs(part_o[slot, h] - ref_o)
            assert np.all(err <= OUT_ATOL + OUT_RTOL * np.abs(ref_o)), \
                f"partial (b={b}, t=[{t0},{t1}), h={h}): max err {err.max()}"
            assert abs(part_lse[slot, h] - ref_l) <= LSE_ATOL, \
                f"partial lse (b={b}, t=[{t0},{t1}), h={h}): {part_lse[slot, h]} vs {ref_l}"
            checked += 1
    assert checked >= splits * int(w["H"])


def test_block_permutation_is_bit_identical(lib, oracle_mod):
    w = spec("perm", 4, 64, 32, [700, 33, 1200, 96], seed=11)
    w2 = wl.permute_blocks(w, seed=5)
    out1, lse1, _ = full_parity(oracle_mod, w)
    out2, lse2, _ = run_library(w2)
    assert np.array_equal(out1, out2) and np.array_equal(lse1, lse2)


def test_repeat_is_deterministic(lib):
    w = spec("det", 5, 128, 32, [2000, 1, 333, 96, 1500], seed=8)
    t = to_device(w)
    out1, lse1, _ = run_library(w, dev_tensors=t)
    out2, lse2, _ = run_library(w, dev_tensors=t)
    assert np.array_equal(out1, out2) and np.array_equal(lse1, lse2)


def test_few_pairs_many_items(lib, oracle_mod):
    # Restrict the grid to 3 CTA pairs so each pair walks a long item list
    # (Q reloads, pipeline carried across items).
    w = spec("few", 9, 128, 32, [100, 2000, 1, 0, 96, 97, 500, 1300, 44], seed=21)
    full_parity(oracle_mod, w, num_clusters=3)


def test_plan_update_and_graph_capture(lib, oracle_mod):
    import torch
    m = lib
    # Cache generated for the longest lengths used below, so every row either
    # plan reads is an N(0,1) token row.
    w = spec("upd", 3, 16, 32, [900, 20, 700], seed=4, max_blocks=32)
    t = to_device(w)
    plan = m.mla_decode_plan(3, 16, np.array([300, 20, 700], dtype=np.int32), 32,
                             int(w["max_blocks"]))
    lens2 = np.array([900, 5, 64], dtype=np.int32)
    w2 = dict(w)
    w2["seq_lens"] = lens2
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        plan.update(lens2, stream)
        t2 = dict(t)
        t2["seq_lens"] = torch.from_numpy(lens2).cuda()
        out = torch.empty((3, 16, 512), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((3, 16), dtype=torch.float32, device="cuda")
        ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device="cuda")
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            m.mla_decode(plan, t2["q_nope"], t2["q_pe"], t2["kv_cache"], t2["block_table"],
                         t2["seq_lens"], float(w["sm_scale"]), out, lse, ws, stream)
        out.fill_(float("nan"))
        g.replay()
    stream.synchronize()
    assert m.mla_check_device_error(plan, stream) == 0
    ref_o, ref_l = oracle_mod.mla_decode(*oracle_args(w2))
    assert_parity(out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
                  ref_o, ref_l, "graph replay")


def test_bad_block_id_sets_error_bit(lib, oracle_mod):
    m = lib
    w = spec("bad", 2, 16, 32, [200, 100], seed=6)
    w["block_table"] = w["block_table"].copy()
    w["block_table"][0, 2] = int(w["num_blocks"]) + 7      # out of range
    out, lse, _ = run_library(w, check_errors=False)
    # no trap, the other request is still right
    ref_o, ref_l = oracle_mod.mla_decode_rows(*oracle_args(spec("bad", 2, 16, 32, [200, 100], seed=6)),
                                              np.array([1] * 16), np.arange(16))
    assert_parity(out[1], lse[1], ref_o, ref_l, "unaffected request")
    # the error is reported on the next check
    plan = m.mla_decode_plan(2, 16, w["seq_lens"], 32, int(w["max_blocks"]))
    t = to_device(w)
    import torch
    o = torch.empty((2, 16, 512), dtype=torch.bfloat16, device="cuda")
    l = torch.empty((2, 16), dtype=torch.float32, device="cuda")
    m.mla_decode(plan, t["q_nope"], t["q_pe"], t["kv_cache"], t["block_table"], t["seq_lens"],
                 float(w["sm_scale"]), o, l)
    assert m.mla_check_device_error(plan) & m.MLA_DEVERR_BAD_BLOCK
    assert m.mla_check_device_error(plan) == 0      # cleared by the read


def test_seq_len_mismatch_sets_error_bit(lib):
    import torch
    m = lib
    w = spec("mm", 2, 16, 32, [200, 100], seed=6)
    t = to_device(w)
    plan = m.mla_decode_plan(2, 16, w["seq_lens"], 32, int(w["max_blocks"]))
    o = torch.empty((2, 16, 512), dtype=torch.bfloat16, device="cuda")
    l = torch.empty((2, 16), dtype=torch.float32, device="cuda")
    bad = torch.tensor([200, 99], dtype=torch.int32, device="cuda")
    m.mla_decode(plan, t["q_nope"], t["q_pe"], t["kv_cache"], t["block_table"], bad,
                 float(w["sm_scale"]), o, l)
    assert m.mla_check_device_error(plan) == m.MLA_DEVERR_SEQLEN_MISMATCH


def test_argument_errors(lib):
    import torch
    m = lib
    w = spec("args", 2, 16, 32, [300, 100], seed=2)
    t = to_device(w)
    plan = m.mla_decode_plan(2, 16, w["seq_lens"], 32, int(w["max_blocks"]), force_splits=2)
    o = torch.empty((2, 16, 512), dtype=torch.bfloat16, device="cuda")
    l = torch.empty((2, 16), dtype=torch.float32, device="cuda")
    args = (t["q_nope"], t["q_pe"], t["kv_cache"], t["block_table"], t["seq_lens"])
    with pytest.raises(m.MLAError) as e:
        m.mla_decode(plan, *args, 0.1, o, l, None)          # workspace required
    assert e.value.status == 3
    small = torch.empty(plan.workspace_bytes - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(m.MLAError):
        m.mla_decode(plan, *args, 0.1, o, l, small)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    with pytest.raises(m.MLAError) as e:
        m.mla_decode(plan, *args, -1.0, o, l, ws)          # sm_scale must be > 0
    assert e.value.status == 1
    for bad in [dict(H=0), dict(H=1025), dict(bs=48)]:
        with pytest.raises(m.MLAError):
            m.mla_decode_plan(2, bad.get("H", 16), w["seq_lens"], bad.get("bs", 32),
                              int(w["max_blocks"]))
    with pytest.raises(m.MLAError):      # longer than the block table allows
        m.mla_decode_plan(2, 16, np.array([10**6, 1]), 32, int(w["max_blocks"]))
    m.mla_decode(plan, *args, 0.1, o, l, ws)
    assert m.mla_check_device_error(plan) == 0


def test_convenience_decode_matches_oracle(lib, oracle_mod):
    """The one-call wrapper (plan from the device lengths, outputs and
    workspace allocated for the caller) on a workload that splits requests."""
    w = wl.generate(wl.WORKLOADS[1])
    t = to_device(w)
    out, lse = lib.decode(t["q_nope"], t["q_pe"], t["kv_cache"], t["block_table"], t["seq_lens"],
                          float(w["sm_scale"]))
    ref_out, ref_lse = oracle_mod.mla_decode(*oracle_args(w))
    assert_parity(out.float().cpu().numpy().astype(np.float64),
                  lse.cpu().numpy().astype(np.float64), ref_out, ref_lse, "decode()")


def test_convenience_decode_multi_token_and_sparse(lib, oracle_mod):
    """decode() with [B, q_len, H, 512] queries and decode_sparse() with a
    top-k list, each allocating its plan, outputs and workspace."""
    import torch
    w = wl.multi_token(wl.custom_spec("api_multi", 3, 32, 32, [40, 300, 97], seed=61), 3)
    t = to_device(w)
    out, lse = lib.decode(t["q_nope"], t["q_pe"], t["kv_cache"], t["block_table"], t["seq_lens"],
                          float(w["sm_scale"]))
    assert tuple(out.shape) == (3, 3, 32, 512) and tuple(lse.shape) == (3, 3, 32)
    ref_out, ref_lse = oracle_mod.mla_decode_multi(w["q_nope"], w["q_pe"], w["kv_cache"],
                                                   w["block_table"], w["seq_lens"], w["sm_scale"])
    assert_parity(out.float().cpu().numpy().astype(np.float64),
                  lse.cpu().numpy().astype(np.float64), ref_out, ref_lse, "decode() q_len=3")
    ws_ = wl.with_topk(spec("api_sparse", 3, 128, 64, [700, 40, 2500], seed=62), 256, seed=63,
                       mixed_padding=True)
    ts = to_device(ws_)
    idx = torch.from_numpy(ws_["topk_indices"]).cuda()
    out, lse = lib.decode_sparse(ts["q_nope"], ts["q_pe"], ts["kv_cache"], ts["block_table"],
                                 ts["seq_lens"], idx, float(ws_["sm_scale"]))
    ref_out, ref_lse = oracle_mod.mla_decode_sparse(ws_["q_nope"], ws_["q_pe"], ws_["kv_cache"],
                                                    ws_["block_table"], ws_["seq_lens"],
                                                    ws_["topk_indices"], ws_["sm_scale"])
    assert_parity(out.float().cpu().numpy().astype(np.float64),
                  lse.cpu().numpy().astype(np.float64), ref_out, ref_lse, "decode_sparse()")


def test_plan_update_growth_keeps_error_word_and_parity(lib, oracle_mod):
    """mla_plan_update on lengths whose schedule outgrows the plan's device
    buffer: the buffer is replaced without a device synchronisation, the
    sticky error word raised before the update is carried over, and a decode
    after the update matches the oracle."""
    import torch
    m = lib
    lens_long = [8000, 7000, 6000]
    w = spec("grow", 3, 32, 32, lens_long, seed=17)
    t = to_device(w)
    short = np.array([10, 3, 1], dtype=np.int32)
    # 64 forced splits: 3 items for the short lengths, 192 for the long ones,
    # so the schedule grows from under 1 KB to over 6 KB (the first device
    # buffer holds 4 KB).
    plan = m.mla_decode_plan(3, 32, short, 32, int(w["max_blocks"]), force_splits=64)
    n_before = plan.num_work_items
    out = torch.empty((3, 32, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((3, 32), dtype=torch.float32, device="cuda")
    # Raise the error word: device lengths that differ from the plan's.
    m.mla_decode(plan, t["q_nope"], t["q_pe"], t["kv_cache"], t["block_table"], t["seq_lens"],
                 float(w["sm_scale"]), out, lse)
    plan.update(np.array(lens_long, dtype=np.int32))
    assert plan.num_work_items > 10 * n_before     # the schedule grew past the old buffer
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device="cuda")
    assert m.mla_check_device_error(plan) == m.MLA_DEVERR_SEQLEN_MISMATCH
    m.mla_decode(plan, t["q_nope"], t["q_pe"], t["kv_cache"], t["block_table"], t["seq_lens"],
                 float(w["sm_scale"]), out, lse, ws)
    assert m.mla_check_device_error(plan) == 0
    ref_o, ref_l = oracle_mod.mla_decode(*oracle_args(w))
    assert_parity(out.float().cpu().numpy().astype(np.float64),
                  lse.cpu().numpy().astype(np.float64), ref_o, ref_l, "after growth")


def test_graph_replay_with_length_bounds(lib, oracle_mod):
    """A plan built for upper bounds on the lengths: one mla_decode captured in
    a CUDA graph, replayed with three different device length vectors (no
    plan update in between), each compared with the oracle. Lengths below a
    split piece's start leave that piece empty (an empty partial)."""
    import torch
    m = lib
    bounds = [1500, 700, 300, 2000, 96]
    w = spec("bounds", 5, 32, 32, bounds, seed=23)
    t = to_device(w)
    plan = m.mla_decode_plan(5, 32, np.array(bounds, dtype=np.int32), 32, int(w["max_blocks"]),
                             num_clusters=8, lengths_are_bounds=True)
    assert any(plan.num_splits(b) > 1 for b in range(5))
    out = torch.empty((5, 32, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((5, 32), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device="cuda")
    lens_dev = torch.tensor(bounds, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        m.mla_decode(plan, t["q_nope"], t["q_pe"], t["kv_cache"], t["block_table"], lens_dev,
                     float(w["sm_scale"]), out, lse, ws, stream)     # warm-up outside capture
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            m.mla_decode(plan, t["q_nope"], t["q_pe"], t["kv_cache"], t["block_table"], lens_dev,
                         float(w["sm_scale"]), out, lse, ws, stream)
    for lens in ([1500, 700, 300, 2000, 96], [1, 650, 0, 1999, 95], [801, 96, 299, 40, 0]):
        lens_dev.copy_(torch.tensor(lens, dtype=torch.int32))
        out.fill_(float("nan"))
        with torch.cuda.stream(stream):
            g.replay()
        stream.synchronize()
        assert m.mla_check_device_error(plan, stream) == 0
        w2 = dict(w)
        w2["seq_lens"] = np.array(lens, dtype=np.int32)
        ref_o, ref_l = oracle_mod.mla_decode(*oracle_args(w2))
        assert_parity(out.float().cpu().numpy().astype(np.float64),
                      lse.cpu().numpy().astype(np.float64), ref_o, ref_l, f"bounds replay {lens}")
    # a length above its bound is reported (and clamped)
    lens_dev.copy_(torch.tensor([1501, 700, 300, 2000, 96], dtype=torch.int32))
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    assert m.mla_check_device_error(plan, stream) == m.MLA_DEVERR_SEQLEN_MISMATCH


def multi_spec(name, B, q_len, H, bs, lens, seed):
    """A workload with q_len query tokens per request: the generator's draws
    for q_len * H rows, viewed as [B, q_len, H, ...]."""
    w = spec(name, B, q_len * H, bs, lens, seed)
    w = dict(w)
    w["q_len"], w["heads"] = q_len, H
    return w


def run_multi(oracle_mod, w, force_splits=0):
    import torch
    m = __import__("paged_mla_decode_05_gb300")
    q_len, H, B = w["q_len"], w["heads"], int(w["B"])
    t = to_device(w)
    plan = m.mla_decode_plan(B, H, w["seq_lens"], int(w["block_size"]), int(w["max_blocks"]),
                             force_splits=force_splits, q_len=q_len)
    qn = t["q_nope"].view(B, q_len, H, 512)
    qp = t["q_pe"].view(B, q_len, H, 64)
    out = torch.full((B, q_len, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, q_len, H), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device="cuda")
    m.mla_decode(plan, qn, qp, t["kv_cache"], t["block_table"], t["seq_lens"],
                 float(w["sm_scale"]), out, lse, ws)
    assert m.mla_check_device_error(plan) == 0
    ref_o, ref_l = oracle_mod.mla_decode_multi(
        w["q_nope"].reshape(B, q_len, H, 512), w["q_pe"].reshape(B, q_len, H, 64), w["kv_cache"],
        w["block_table"], w["seq_lens"], w["sm_scale"])
    assert_parity(out.float().cpu().numpy().astype(np.float64),
                  lse.cpu().numpy().astype(np.float64), ref_o, ref_l,
                  f"{w['name']} q_len={q_len}")
    return plan


@pytest.mark.parametrize("q_len", [2, 4])
def test_multi_token_v2lite_shape(lib, oracle_mod, q_len):
    """Speculative decoding on the DeepSeek-V2-Lite shape (B=64, H=16,
    lengths U{q_len..4096}, block size 64): every element against the oracle."""
    lens = np.random.default_rng(40 + q_len).integers(q_len, 4096, size=64, endpoint=True)
    run_multi(oracle_mod, multi_spec("v2lite_multi", 64, q_len, 16, 64, lens.tolist(), seed=q_len))


@pytest.mark.parametrize("q_len", [2, 4])
def test_multi_token_r1_shape(lib, oracle_mod, q_len):
    """Speculative decoding on the DeepSeek-R1 shape (H=128: q_len * 128 query
    rows per request in head groups of 128), lengths 1024 + U{0..2048}."""
    lens = 1024 + np.random.default_rng(50 + q_len).integers(0, 2048, size=16, endpoint=True)
    run_multi(oracle_mod, multi_spec("r1_multi", 16, q_len, 128, 32, lens.tolist(), seed=q_len))


def test_multi_token_split_pieces_with_empty_rows(lib, oracle_mod):
    """Forced splits put a piece of request 1 at tokens [576, 577), where the
    first three of its four query tokens see no token: their partials are
    empty (lse = -inf) and the combine must ignore them."""
    w = multi_spec("multi_split", 3, 4, 16, 32, [4, 577, 300], seed=3)
    plan = run_multi(oracle_mod, w, force_splits=7)
    assert plan.num_splits(1) == 7
