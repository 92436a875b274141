"""GPU parity of the sm_103a decode (through the C ABI) against the fp64 oracle.

Small and medium workloads are compared element by element over every
(request, head); the largest ones on sampled rows the oracle computes one by
one, in the same launch configuration the benchmark times.
"""
import numpy as np
import pytest

import mla_workloads as wl
from gpu_helpers import (assert_parity, oracle_args, run_library, sample_rows, spec, to_device)

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


@pytest.mark.parametrize("idx,n_random,full", [(2, 96, (0, 77)), (3, 96, (5, 400)),
                                               (4, 0, (0, 1, 2, 3))])
def test_large_configs_sampled(lib, oracle_mod, idx, n_random, full):
    w = wl.generate(wl.WORKLOADS[idx])
    out, lse, plan = run_library(w)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    rb, rh = sample_rows(w, n_random, seed=idx, full_requests=full)
    ref_o, ref_l = oracle_mod.mla_decode_rows(*oracle_args(w), rb, rh)
    assert_parity(out[rb, rh], lse[rb, rh], ref_o, ref_l, w["name"])
    if idx == 4:   # the 64K request must be split across pairs and recombined
        assert plan.num_splits(0) > 1


@pytest.mark.parametrize("H", [1, 7, 32, 100, 128])
def test_head_counts(lib, oracle_mod, H):
    full_parity(oracle_mod, spec(f"h{H}", 3, H, 32, [1, 97, 300], seed=H))


@pytest.mark.parametrize("bs", [16, 32, 64, 128])
def test_block_sizes_ragged(lib, oracle_mod, bs):
    lens = [1, 15, 95, 96, 97, 191, 192, 193, 500]
    full_parity(oracle_mod, spec(f"bs{bs}", len(lens), 16, bs, lens, seed=bs))


def test_empty_and_tiny_requests(lib, oracle_mod):
    w = spec("empty", 4, 8, 32, [0, 1, 0, 2], seed=3)
    out, lse, _ = full_parity(oracle_mod, w)
    assert np.all(out[0] == 0) and np.all(lse[0] == -np.inf)


@pytest.mark.parametrize("splits", [2, 3, 7])
def test_forced_splits_match_oracle_and_unsplit(lib, oracle_mod, splits):
    w = spec("split", 3, 128, 64, [1000, 96 * 5 + 1, 50], seed=splits, peaky_fraction=0.02)
    out1, lse1, _ = full_parity(oracle_mod, w)
    out2, lse2, plan = full_parity(oracle_mod, w, force_splits=splits)
    assert plan.num_splits(0) == splits and plan.workspace_bytes > 0
    # Split invariance: both partitions are within the parity tolerance of the
    # oracle, so they agree within twice that bound (they differ by the fp32
    # summation order, the bf16 rounding of P relative to each split's own
    # running max, and one bf16 rounding of out).
    assert np.all(np.abs(out1 - out2) <= 2 * (2e-2 + 2e-2 * np.abs(out1)))
    assert np.max(np.abs(lse1 - lse2)) < 2 * 5e-3


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
    for bad in [dict(H=0), dict(H=129), dict(bs=48)]:
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
