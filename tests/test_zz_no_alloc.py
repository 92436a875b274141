"""mla_decode_no_alloc, the entry point for callers that cannot allocate device
memory while they decode (an engine whose caching allocator owns nearly all of
HBM, or a host thread that must not stall on cudaMalloc's synchronisation).

It runs the same kernels as mla_decode with its workspace, work list and error
word in the library's fixed device scratch. The GPU test makes two calls in a
row, so the second runs on the scratch the first left behind, and checks each
against mla_decode on the same inputs under the parity tolerance of the other
GPU tests. This file sorts last so that a run stopping at the first failure has
run every other test before it.
"""
import ctypes

import numpy as np
import pytest

import mla_workloads as wl
from gpu_helpers import LSE_ATOL, OUT_ATOL, OUT_RTOL, run_library, to_device

SCRATCH_BYTES = 32 << 20  # MLA_NO_ALLOC_SCRATCH_BYTES


@pytest.fixture(scope="module")
def m():
    from paged_mla_decode_05_gb300 import build
    build.build()
    import paged_mla_decode_05_gb300 as mod
    return mod


def _no_alloc(m, w, t):
    """One mla_decode_no_alloc call with a host-only plan (no device memory
    allocated by planning either); returns out, lse as float64 and the bits."""
    import torch
    B, H = int(w["B"]), int(w["H"])
    plan = m.mla_decode_plan(B, H, w["seq_lens"], int(w["block_size"]), int(w["max_blocks"]),
                             host_only=True)
    out = torch.full((B, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
    bits = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    m.mla_decode_no_alloc(plan, t["q_nope"], t["q_pe"], t["kv_cache"], t["block_table"],
                          t["seq_lens"], float(w["sm_scale"]), out, lse, bits)
    torch.cuda.synchronize()
    return (out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
            int(bits.item()), plan)


@pytest.mark.gpu
def test_two_calls_in_a_row_match_mla_decode(m):
    # Both workloads split requests, so both calls write and read partials in
    # the scratch; the second (H = 128, 75 slots, about 19 MiB) overwrites
    # what the first (H = 16, 115 slots) left there.
    for name in ("v2lite_b64_h16", "long_b4_h128"):
        w = wl.generate(wl.WORKLOADS_BY_NAME[name])
        t = to_device(w)
        out, lse, bits, plan = _no_alloc(m, w, t)
        assert plan.workspace_bytes > 0, f"{name}: expected split partials"
        assert bits == 0, f"{name}: device error bits {bits}"
        ref_out, ref_lse, _ = run_library(w, dev_tensors=t)
        assert np.all(np.isfinite(out)), f"{name}: non-finite output"
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.isfinite(lse), fin), f"{name}: lse finiteness differs"
        err = np.abs(out - ref_out)
        assert (err <= OUT_ATOL + OUT_RTOL * np.abs(ref_out)).all(), \
            f"{name}: max |out - mla_decode| = {err.max()}"
        lerr = np.abs(lse[fin] - ref_lse[fin])
        assert lerr.size == 0 or lerr.max() <= LSE_ATOL, f"{name}: lse error {lerr.max()}"
        print(f"[no-alloc] {name}: max|out diff|={err.max():.3g} max|lse diff|="
              f"{lerr.max() if lerr.size else 0:.3g}")


def test_plan_beyond_the_scratch_is_refused(m):
    # 8 requests x 32 forced splits x 128 heads of fp32 partials = 67 MB, more
    # than the scratch holds; the call refuses it before touching any device.
    lens = np.full(8, 65536, dtype=np.int32)
    plan = m.mla_decode_plan(8, 128, lens, 64, 1024, num_clusters=76, force_splits=32,
                             host_only=True)
    assert plan.workspace_bytes > SCRATCH_BYTES
    fake = ctypes.c_void_p(256)
    rc = m._lib.LIB.mla_decode_no_alloc(plan.handle, fake, fake, fake, 1 << 16, fake, fake,
                                        ctypes.c_float(0.07), fake, fake, None, None)
    assert rc == 3, m.mla_status_string(rc)  # MLA_ERR_WORKSPACE_TOO_SMALL
