"""mla_decode_no_alloc, the entry point for callers that cannot allocate device
memory while they decode (an engine whose caching allocator owns nearly all of
HBM, or a host thread that must not stall on cudaMalloc's synchronisation).

It runs the same kernels as mla_decode with its workspace and work list in the
library's fixed device scratch. The GPU test makes three calls in a row, so
each runs on the scratch the previous one left behind; the third uses fewer
bytes of partials than the second, so the second's leftovers stay in the
scratch around what the third reads. Each call is checked against the fp64
oracle and against mla_decode on the same inputs, under the parity tolerance
of the other GPU tests. This file sorts last so that a run stopping at the
first failure has run every other test before it.
"""
import ctypes

import numpy as np
import pytest

import mla_workloads as wl
from gpu_helpers import assert_parity, oracle_args, run_library, spec, to_device

SCRATCH_BYTES = 32 << 20  # MLA_NO_ALLOC_SCRATCH_BYTES


@pytest.fixture(scope="module")
def m():
    from paged_mla_decode_05_gb300 import build
    build.build()
    import paged_mla_decode_05_gb300 as mod
    return mod


def _no_alloc(m, w, t, force_splits=0):
    """One mla_decode_no_alloc call with a host-only plan (no device memory
    allocated by planning either); returns out, lse as float64, the error
    bits and the plan."""
    import torch
    B, H = int(w["B"]), int(w["H"])
    plan = m.mla_decode_plan(B, H, w["seq_lens"], int(w["block_size"]), int(w["max_blocks"]),
                             host_only=True, force_splits=force_splits)
    out = torch.full((B, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
    bits = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    m.mla_decode_no_alloc(plan, t["q_nope"], t["q_pe"], t["kv_cache"], t["block_table"],
                          t["seq_lens"], float(w["sm_scale"]), out, lse, bits)
    torch.cuda.synchronize()
    return (out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
            int(bits.item()), plan)


def _partial_bytes(plan):
    items = plan.work_items()
    slots = sum(1 for it in items if it[3] >= 0)
    return slots * plan.H * 512 * 4


@pytest.mark.gpu
def test_three_calls_in_a_row_match_oracle_and_mla_decode(m, oracle_mod):
    # All three workloads split requests, so every call writes and reads
    # partials in the scratch. The second (H = 128, 75 slots, about 19 MiB)
    # overwrites what the first (H = 16, 115 slots) left; the third (H = 128,
    # two forced splits of a 300-token request, 0.5 MiB) reads only the start
    # of the region the second filled.
    cases = [(wl.generate(wl.WORKLOADS_BY_NAME["v2lite_b64_h16"]), 0),
             (wl.generate(wl.WORKLOADS_BY_NAME["long_b4_h128"]), 0),
             (spec("after_long", 3, 128, 32, [300, 1, 77], seed=13), 2)]
    sizes = []
    for w, splits in cases:
        name = w["name"]
        t = to_device(w)
        out, lse, bits, plan = _no_alloc(m, w, t, force_splits=splits)
        assert plan.workspace_bytes > 0, f"{name}: expected split partials"
        assert bits == 0, f"{name}: device error bits {bits}"
        ref_out, ref_lse = oracle_mod.mla_decode(*oracle_args(w))
        assert_parity(out, lse, ref_out, ref_lse, f"no-alloc {name} vs oracle")
        lib_out, lib_lse, _ = run_library(w, dev_tensors=t, force_splits=splits)
        assert_parity(out, lse, lib_out, lib_lse, f"no-alloc {name} vs mla_decode")
        sizes.append(_partial_bytes(plan))
    assert sizes[2] < sizes[1], "the third call must leave the second's partials around it"


@pytest.mark.gpu
def test_refuses_stream_capture_and_null_error_word(m):
    import torch
    w = spec("cap", 2, 16, 32, [100, 5], seed=3)
    t = to_device(w)
    plan = m.mla_decode_plan(2, 16, w["seq_lens"], 32, int(w["max_blocks"]), host_only=True)
    out = torch.empty((2, 16, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((2, 16), dtype=torch.float32, device="cuda")
    bits = torch.zeros((1,), dtype=torch.int32, device="cuda")
    args = (t["q_nope"], t["q_pe"], t["kv_cache"], t["block_table"], t["seq_lens"],
            float(w["sm_scale"]), out, lse)
    # An ordinary call first: the entry point's one-time set-up on this device
    # happens outside any capture.
    m.mla_decode_no_alloc(plan, *args, bits)
    torch.cuda.synchronize()
    assert int(bits.item()) == 0
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with pytest.raises(m.MLAError) as e:
            with torch.cuda.graph(g, stream=stream):
                m.mla_decode_no_alloc(plan, *args, bits, stream)
    assert e.value.status == 1   # MLA_ERR_INVALID_ARG, nothing enqueued
    rc = m._lib.LIB.mla_decode_no_alloc(plan.handle, *(ctypes.c_void_p(a.data_ptr()) for a in
                                                         (t["q_nope"], t["q_pe"], t["kv_cache"])),
                                        int(w["num_blocks"]), ctypes.c_void_p(t["block_table"].data_ptr()),
                                        ctypes.c_void_p(t["seq_lens"].data_ptr()),
                                        ctypes.c_float(0.07), ctypes.c_void_p(out.data_ptr()),
                                        ctypes.c_void_p(lse.data_ptr()), None, None)
    assert rc == 1, m.mla_status_string(rc)
    # The device is still usable and the entry point still works afterwards.
    m.mla_decode_no_alloc(plan, *args, bits)
    torch.cuda.synchronize()
    assert int(bits.item()) == 0


def test_plan_beyond_the_scratch_is_refused(m):
    # 8 requests x 32 forced splits x 128 heads of fp32 partials = 67 MB, more
    # than the scratch holds; the call refuses it before touching any device.
    lens = np.full(8, 65536, dtype=np.int32)
    plan = m.mla_decode_plan(8, 128, lens, 64, 1024, num_clusters=76, force_splits=32,
                             host_only=True)
    assert plan.workspace_bytes > SCRATCH_BYTES
    fake = ctypes.c_void_p(256)
    rc = m._lib.LIB.mla_decode_no_alloc(plan.handle, fake, fake, fake, 1 << 16, fake, fake,
                                        ctypes.c_float(0.07), fake, fake, fake, None)
    assert rc == 3, m.mla_status_string(rc)  # MLA_ERR_WORKSPACE_TOO_SMALL
    rc = m._lib.LIB.mla_decode_no_alloc(plan.handle, fake, fake, fake, 1 << 16, fake, fake,
                                        ctypes.c_float(0.07), fake, fake, None, None)
    assert rc == 1, m.mla_status_string(rc)  # a NULL error word is refused first
