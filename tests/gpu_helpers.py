"""Helpers shared by the GPU tests: run the library on seeded inputs and compare
with the oracle under the parity tolerance.

Tolerance (fixed for this method): |out - ref| <= 2e-2 + 2e-2 |ref| per
element, |lse - ref| <= 5e-3, every value finite. The kernels round P to bf16
(FP8 cache: two E4M3 terms, about as fine) before P.V and round out to bf16
(relative 2^-9), which the bound covers with room to spare. The FP8 oracle
reads the same E4M3 bytes exactly, so the cache's own quantisation is not
part of the error.
"""
import numpy as np

import mla_workloads as wl

OUT_ATOL = 2e-2
OUT_RTOL = 2e-2
LSE_ATOL = 5e-3


def to_device(w):
    import torch
    dev = torch.device("cuda", 0)

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    t = {
        "q_nope": bf16(w["q_nope"]),
        "q_pe": bf16(w["q_pe"]),
        "block_table": torch.from_numpy(np.ascontiguousarray(w["block_table"])).to(dev),
        "seq_lens": torch.from_numpy(np.ascontiguousarray(w["seq_lens"])).to(dev),
    }
    if "kv_fp8" in w:   # FP8 workload (mla_workloads.to_fp8): E4M3 bytes
        t["kv_fp8"] = torch.from_numpy(np.ascontiguousarray(w["kv_fp8"])).to(dev)
    else:
        t["kv_cache"] = bf16(w["kv_cache"])
    return t


def decode_into(m, plan, w, t, qn, qp, out, lse, ws):
    """mla_decode, or mla_decode_fp8 for an FP8 workload."""
    if "kv_fp8" in w:
        m.mla_decode_fp8(plan, qn, qp, t["kv_fp8"], float(w["kv_scale"]), t["block_table"],
                         t["seq_lens"], float(w["sm_scale"]), out, lse, ws)
    else:
        m.mla_decode(plan, qn, qp, t["kv_cache"], t["block_table"], t["seq_lens"],
                     float(w["sm_scale"]), out, lse, ws)


def oracle_ref(oracle_mod, w):
    """The oracle's (out, lse) for a bf16 or an FP8 workload."""
    if "kv_fp8" in w:
        return oracle_mod.mla_decode_fp8(w["q_nope"], w["q_pe"], w["kv_fp8"], w["kv_scale"],
                                         w["block_table"], w["seq_lens"], w["sm_scale"])
    return oracle_mod.mla_decode(*oracle_args(w))


def run_library(w, force_splits=0, num_clusters=0, dev_tensors=None, check_errors=True):
    """Plan + decode through the C ABI; returns (out f64 [B,H,512], lse f64 [B,H], plan)."""
    import torch
    import paged_mla_decode_05_gb300 as m
    t = dev_tensors if dev_tensors is not None else to_device(w)
    B, H = int(w["B"]), int(w["H"])
    plan = m.mla_decode_plan(B, H, w["seq_lens"], int(w["block_size"]), int(w["max_blocks"]),
                             num_clusters=num_clusters, force_splits=force_splits)
    out = torch.full((B, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
    ws = None
    if plan.workspace_bytes:
        ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    decode_into(m, plan, w, t, t["q_nope"], t["q_pe"], out, lse, ws)
    bits = m.mla_check_device_error(plan)
    if check_errors:
        assert bits == 0, f"device error bits {bits}"
    out_np = out.float().cpu().numpy().astype(np.float64)
    lse_np = lse.cpu().numpy().astype(np.float64)
    return out_np, lse_np, plan


def assert_parity(out, lse, ref_out, ref_lse, what=""):
    assert np.all(np.isfinite(out)), f"{what}: non-finite output"
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin), f"{what}: lse finiteness differs"
    err = np.abs(out - ref_out)
    bound = OUT_ATOL + OUT_RTOL * np.abs(ref_out)
    bad = err > bound
    if bad.any():
        idx = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} output elements out of tolerance; worst "
                             f"at {idx}: got {out[idx]} ref {ref_out[idx]}")
    lerr = np.abs(lse[fin] - ref_lse[fin])
    assert lerr.size == 0 or lerr.max() <= LSE_ATOL, f"{what}: lse error {lerr.max()}"
    margin = float((err / bound).max()) if err.size else 0.0
    print(f"[parity] {what}: max|out-ref|={err.max() if err.size else 0:.3g} "
          f"(max fraction of tolerance {margin:.3f}), max|lse-ref|="
          f"{lerr.max() if lerr.size else 0:.3g}")
    return float(err.max()), float(lerr.max()) if lerr.size else 0.0


def oracle_args(w):
    return (w["q_nope"], w["q_pe"], w["kv_cache"], w["block_table"], w["seq_lens"], w["sm_scale"])


def spec(name, B, H, bs, lens, seed, **kw):
    return wl.generate(wl.custom_spec(name, B=B, H=H, block_size=bs, seq_lens=lens, seed=seed, **kw))
