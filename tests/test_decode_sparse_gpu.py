"""GPU parity of the sparse (top-k) decode (mla_sparse_plan + mla_decode_sparse,
through the C ABI) against the oracle's sparse decode on the same inputs.

Each request attends only to the tokens its row of topk_indices lists; an
entry outside [0, L) is padding and a listed token counts once per listing.
The bf16 and FP8 caches are both covered, at the B=64, H=128, top-2048
workload the benchmark times and on small edge cases (short and empty lists,
padding between selected tokens, duplicates, head groups, a CUDA graph
replayed with new lists and lengths).
"""
import numpy as np
import pytest

import mla_workloads as wl
from gpu_helpers import assert_parity, spec

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


def _dev(w):
    import torch
    dev = torch.device("cuda", 0)

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    t = {"q_nope": bf16(w["q_nope"]), "q_pe": bf16(w["q_pe"]),
         "block_table": torch.from_numpy(np.ascontiguousarray(w["block_table"])).to(dev),
         "seq_lens": torch.from_numpy(np.ascontiguousarray(w["seq_lens"])).to(dev),
         "topk_indices": torch.from_numpy(np.ascontiguousarray(w["topk_indices"])).to(dev)}
    if "kv_fp8" in w:
        t["kv"] = torch.from_numpy(np.ascontiguousarray(w["kv_fp8"])).to(dev)
    else:
        t["kv"] = bf16(w["kv_cache"])
    return t


def _oracle(oracle_mod, w):
    if "kv_fp8" in w:
        return oracle_mod.mla_decode_sparse(w["q_nope"], w["q_pe"], None, w["block_table"],
                                            w["seq_lens"], w["topk_indices"], w["sm_scale"],
                                            kv_fp8=w["kv_fp8"], kv_scale=w["kv_scale"])
    return oracle_mod.mla_decode_sparse(w["q_nope"], w["q_pe"], w["kv_cache"], w["block_table"],
                                        w["seq_lens"], w["topk_indices"], w["sm_scale"])


def run_sparse(m, w, t=None, check_errors=True, **plan_kw):
    import torch
    t = t if t is not None else _dev(w)
    B, H = int(w["B"]), int(w["H"])
    topk = int(w["topk_indices"].shape[1])
    plan = m.mla_sparse_plan(B, H, topk, **plan_kw)
    out = torch.full((B, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    m.mla_decode_sparse(plan, t["q_nope"], t["q_pe"], t["kv"], t["block_table"], t["seq_lens"],
                        t["topk_indices"], float(w["sm_scale"]), out, lse, ws,
                        kv_scale=float(w["kv_scale"]) if "kv_fp8" in w else None)
    bits = m.mla_check_device_error(plan)
    if check_errors:
        assert bits == 0, f"device error bits {bits}"
    return (out.float().cpu().numpy().astype(np.float64),
            lse.cpu().numpy().astype(np.float64), plan, bits)


def sparse_parity(m, oracle_mod, w, what, **plan_kw):
    out, lse, plan, _ = run_sparse(m, w, **plan_kw)
    ref_out, ref_lse = _oracle(oracle_mod, w)
    assert_parity(out, lse, ref_out, ref_lse, what)
    return plan


def _bench_workload(seed=6):
    w = wl.generate(wl.SPARSE_WORKLOADS["sparse_r1_b64_h128"])
    return wl.with_topk(w, wl.SPARSE_TOPK, seed=seed)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_sparse_r1_b64_top2048_full(lib, oracle_mod, kv):
    """Every (request, head) of the B=64, H=128, top-2048 workload, in the
    launch configuration the benchmark times."""
    w = _bench_workload()
    if kv == "fp8":
        w = wl.to_fp8(w)
    sparse_parity(lib, oracle_mod, w, f"sparse_r1_b64_h128 {kv}")


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_sparse_mixed_padding_and_short_requests(lib, oracle_mod, kv):
    """Requests shorter than topk (fewer valid entries), empty ones, and
    padding (-1 and positions past L) scattered between selected tokens."""
    w = spec("sp_pad", 7, 128, 64, [0, 1, 5, 63, 64, 65, 3000], seed=41)
    w = wl.with_topk(w, 96, seed=42, mixed_padding=True)
    if kv == "fp8":
        w = wl.to_fp8(w)
    sparse_parity(lib, oracle_mod, w, f"sparse mixed padding {kv}")


@pytest.mark.parametrize("topk", [1, 7, 31, 32, 33, 96, 97, 300, 4096])
def test_sparse_topk_values(lib, oracle_mod, topk):
    """Lists of every length class: below, at and past a 32-row piece, a tile
    (96) and a 64-position plan block; 4096 is longer than every request."""
    w = spec(f"sp_k{topk}", 4, 128, 32, [500, 1, 97, 3000], seed=topk)
    w = wl.with_topk(w, topk, seed=topk + 1)
    sparse_parity(lib, oracle_mod, w, f"sparse topk={topk}")


@pytest.mark.parametrize("bs", [16, 32, 64, 128])
def test_sparse_source_block_sizes(lib, oracle_mod, bs):
    w = spec(f"sp_bs{bs}", 3, 64, bs, [bs * 7 + 3, 2 * bs - 1, 1000], seed=50 + bs)
    w = wl.with_topk(w, 200, seed=bs, mixed_padding=True)
    sparse_parity(lib, oracle_mod, w, f"sparse bs={bs}")


@pytest.mark.parametrize("H", [16, 100, 192])
def test_sparse_head_counts(lib, oracle_mod, H):
    """16 and 100 heads (a group padded inside the kernel) and 192 (two head
    groups over the same row list)."""
    w = spec(f"sp_h{H}", 3, H, 64, [700, 40, 2500], seed=H)
    w = wl.with_topk(w, 256, seed=H + 3)
    sparse_parity(lib, oracle_mod, w, f"sparse H={H}")


@pytest.mark.parametrize("H", [16, 192])
def test_sparse_fp8_head_counts(lib, oracle_mod, H):
    """FP8 cache with a padded head group and with two head groups."""
    w = spec(f"sp8_h{H}", 3, H, 64, [700, 40, 2500], seed=H + 11)
    w = wl.to_fp8(wl.with_topk(w, 256, seed=H + 13, mixed_padding=True))
    sparse_parity(lib, oracle_mod, w, f"sparse fp8 H={H}")


def test_sparse_fp8_forced_splits(lib, oracle_mod):
    w = spec("sp8_split", 2, 128, 64, [5000, 3000], seed=98)
    w = wl.to_fp8(wl.with_topk(w, 2048, seed=99))
    plan = sparse_parity(lib, oracle_mod, w, "sparse fp8 forced splits", force_splits=3)
    assert plan.num_splits(1) == 3


def test_sparse_duplicates_count_twice(lib, oracle_mod):
    w = spec("sp_dup", 2, 128, 64, [300, 90], seed=77)
    idx = np.array([[5, 5, 5, 299, 0, 17, 17, -1, 100, 101],
                    [89, 0, 0, 44, 44, 44, 44, 90, -3, 12]], dtype=np.int32)
    w = dict(w)
    w["topk_indices"] = idx
    sparse_parity(lib, oracle_mod, w, "sparse duplicates")


def test_sparse_forced_splits(lib, oracle_mod):
    """A plan that splits each list across CTA pairs (combine kernel path)."""
    w = spec("sp_split", 2, 128, 64, [5000, 3000], seed=88)
    w = wl.with_topk(w, 2048, seed=89)
    plan = sparse_parity(lib, oracle_mod, w, "sparse forced splits", force_splits=4)
    assert plan.num_splits(0) == 4


def test_sparse_bad_block_id_is_reported_and_skipped(lib, oracle_mod):
    """A selected token whose page id lies outside the pool is not read: the
    device error bit MLA_DEVERR_BAD_BLOCK is set and the token is dropped."""
    import torch
    w = spec("sp_bad", 2, 128, 64, [640, 640], seed=91)
    w = wl.with_topk(w, 128, seed=92)
    bad_page = int(w["topk_indices"][1, 0]) // 64
    bt = np.array(w["block_table"], copy=True)
    bt[1, bad_page] = 1 << 30
    t = _dev(w)
    t["block_table"].copy_(torch.from_numpy(bt))
    out, lse, _, bits = run_sparse(lib, w, t=t, check_errors=False)
    assert bits & 1
    # the oracle sees the good table and request 1's list without that page
    idx = np.array(w["topk_indices"], copy=True)
    idx[1][idx[1] // 64 == bad_page] = -1
    ref_out, ref_lse = _oracle(oracle_mod, dict(w, topk_indices=idx))
    assert_parity(out, lse, ref_out, ref_lse, "sparse bad block")


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_sparse_graph_replay_with_new_lists(lib, oracle_mod, kv):
    """One captured CUDA graph serves new lists and new lengths: the plan is
    built for topk alone, the lists and lengths are read on the device."""
    import torch
    m = lib
    lens = [3000, 200, 1500]
    w0 = wl.with_topk(spec("sp_graph", 3, 128, 64, lens, seed=93), 512, seed=0)
    if kv == "fp8":
        w0 = wl.to_fp8(w0)
    kv_scale = float(w0["kv_scale"]) if kv == "fp8" else None
    t = _dev(w0)
    B, H, topk = 3, 128, 512
    plan = m.mla_sparse_plan(B, H, topk)
    out = torch.empty((B, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        m.mla_decode_sparse(plan, t["q_nope"], t["q_pe"], t["kv"], t["block_table"],
                            t["seq_lens"], t["topk_indices"], float(w0["sm_scale"]), out, lse,
                            ws, kv_scale=kv_scale, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        m.mla_decode_sparse(plan, t["q_nope"], t["q_pe"], t["kv"], t["block_table"],
                            t["seq_lens"], t["topk_indices"], float(w0["sm_scale"]), out, lse,
                            ws, kv_scale=kv_scale, stream=s)
    for step, new_lens in enumerate([lens, [2999, 0, 1501], [64, 192, 1]]):
        w = dict(w0)
        w["seq_lens"] = np.array(new_lens, dtype=np.int32)
        w = wl.with_topk(w, topk, seed=10 + step, mixed_padding=step == 2)
        t["seq_lens"].copy_(torch.from_numpy(w["seq_lens"]))
        t["topk_indices"].copy_(torch.from_numpy(w["topk_indices"]))
        g.replay()
        torch.cuda.synchronize()
        assert m.mla_check_device_error(plan) == 0
        ref_out, ref_lse = _oracle(oracle_mod, w)
        assert_parity(out.float().cpu().numpy().astype(np.float64),
                      lse.cpu().numpy().astype(np.float64), ref_out, ref_lse,
                      f"sparse graph replay {kv} {step}")


def test_sparse_argument_errors(lib):
    import torch
    m = lib
    w = wl.with_topk(spec("sp_args", 2, 128, 64, [100, 50], seed=95), 64, seed=1)
    t = _dev(w)
    sparse = m.mla_sparse_plan(2, 128, 64)
    dense = m.mla_decode_plan(2, 128, w["seq_lens"], 64, int(w["max_blocks"]))
    out = torch.empty((2, 128, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((2, 128), dtype=torch.float32, device="cuda")
    ws = torch.empty(sparse.workspace_bytes, dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):   # a dense plan has no list length
        m.mla_decode_sparse(dense, t["q_nope"], t["q_pe"], t["kv"], t["block_table"],
                            t["seq_lens"], t["topk_indices"], 0.1, out, lse, ws)
    with pytest.raises(m.MLAError):   # a sparse plan does not serve the dense call
        m.mla_decode(sparse, t["q_nope"], t["q_pe"], t["kv"],
                     t["block_table"][:, :sparse.max_blocks].contiguous(), t["seq_lens"], 0.1,
                     out, lse, ws)
    with pytest.raises(m.MLAError):   # workspace too small
        m.mla_decode_sparse(sparse, t["q_nope"], t["q_pe"], t["kv"], t["block_table"],
                            t["seq_lens"], t["topk_indices"], 0.1, out, lse,
                            ws[:sparse.workspace_bytes - 1])
    with pytest.raises(ValueError):   # list of the wrong length
        m.mla_decode_sparse(sparse, t["q_nope"], t["q_pe"], t["kv"], t["block_table"],
                            t["seq_lens"], t["topk_indices"][:, :32].contiguous(), 0.1, out,
                            lse, ws)
    torch.cuda.synchronize()
