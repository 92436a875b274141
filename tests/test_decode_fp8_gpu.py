"""GPU parity of the FP8-cache decode (mla_decode_fp8, through the C ABI)
against the fp64 oracle on the same E4M3 bytes.

Every workload, the B=512, H=128 one the benchmark times included, is
converted to an FP8 cache (mla_workloads.to_fp8: E4M3 of element / 0.1) and
compared element by element over every (request, head) under the parity
tolerance, in the launch configuration the benchmark uses.
"""
import numpy as np
import pytest

import mla_workloads as wl
from gpu_helpers import assert_parity, oracle_ref, run_library, spec, to_device

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


def fp8_parity(oracle_mod, w, **kw):
    w8 = wl.to_fp8(w)
    out, lse, plan = run_library(w8, **kw)
    ref_out, ref_lse = oracle_ref(oracle_mod, w8)
    assert_parity(out, lse, ref_out, ref_lse, w8["name"])
    return out, lse, plan


@pytest.mark.parametrize("idx", [0, 1, 2, 3, 4])
def test_fp8_configs_full(lib, oracle_mod, idx):
    """The five workloads with an FP8 cache: tiny, V2-Lite (16 heads, padded
    inside the kernel), R1 B=128, R1 B=512 and the long-context split one."""
    w = wl.generate(wl.WORKLOADS[idx])
    _, _, plan = fp8_parity(oracle_mod, w)
    if idx == 4:
        assert plan.num_splits(0) > 1


@pytest.mark.parametrize("H", [1, 7, 100, 128, 192])
def test_fp8_head_counts(lib, oracle_mod, H):
    fp8_parity(oracle_mod, spec(f"f8h{H}", 3, H, 32, [1, 97, 300], seed=100 + H))


@pytest.mark.parametrize("bs", [16, 32, 64, 128])
def test_fp8_block_sizes_ragged(lib, oracle_mod, bs):
    fp8_parity(oracle_mod, spec(f"f8bs{bs}", 4, 32, bs, [1, bs - 1, 3 * bs + 5, 1000], seed=bs))


def test_fp8_empty_and_tiny_requests(lib, oracle_mod):
    fp8_parity(oracle_mod, spec("f8edge", 6, 16, 32, [0, 1, 2, 95, 96, 97], seed=9))


@pytest.mark.parametrize("splits", [2, 7])
def test_fp8_forced_splits(lib, oracle_mod, splits):
    w = spec(f"f8split{splits}", 3, 64, 32, [5, 700, 2000], seed=splits, peaky_fraction=0.02)
    _, _, plan = fp8_parity(oracle_mod, w, force_splits=splits)
    assert plan.num_splits(2) == splits


def test_fp8_query_rows_of_very_different_magnitude(lib, oracle_mod):
    """Q rows scaled by 2^12, 2^-12 and 0: each row's power-of-two scale of
    the two-term Q split follows its own magnitude."""
    w = spec("f8qscale", 2, 8, 32, [300, 41], seed=21)
    w = dict(w)
    qn = wl.bf16_bits_to_f32(w["q_nope"]).copy()
    qp = wl.bf16_bits_to_f32(w["q_pe"]).copy()
    for h, f in ((1, 2.0 ** 12), (2, 2.0 ** -12), (3, 0.0), (5, 2.0 ** 6)):
        qn[:, h] *= np.float32(f)
        qp[:, h] *= np.float32(f)
    w["q_nope"] = wl.f32_to_bf16_bits(qn)
    w["q_pe"] = wl.f32_to_bf16_bits(qp)
    w["sm_scale"] = 1.0 / 4096.0   # keeps the 2^12 rows' scores finite and moderate
    fp8_parity(oracle_mod, w)


def test_fp8_block_permutation_is_bit_identical(lib):
    w8 = wl.to_fp8(spec("f8perm", 4, 32, 16, [33, 180, 7, 500], seed=5))
    a = run_library(w8)
    b = run_library(wl.permute_blocks(w8, seed=11))
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_fp8_multi_token(lib, oracle_mod):
    """Speculative decoding (q_len = 3) over an FP8 cache, with forced splits."""
    import torch
    m = lib
    q_len, H, B = 3, 16, 3
    w = wl.to_fp8(spec("f8multi", B, q_len * H, 32, [3, 577, 1200], seed=31))
    t = to_device(w)
    plan = m.mla_decode_plan(B, H, w["seq_lens"], 32, int(w["max_blocks"]), force_splits=3,
                             q_len=q_len)
    qn = t["q_nope"].view(B, q_len, H, 512)
    qp = t["q_pe"].view(B, q_len, H, 64)
    out = torch.full((B, q_len, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, q_len, H), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device="cuda")
    m.mla_decode_fp8(plan, qn, qp, t["kv_fp8"], w["kv_scale"], t["block_table"], t["seq_lens"],
                     float(w["sm_scale"]), out, lse, ws)
    assert m.mla_check_device_error(plan) == 0
    ref_o, ref_l = oracle_mod.mla_decode_fp8(
        w["q_nope"].reshape(B, q_len, H, 512), w["q_pe"].reshape(B, q_len, H, 64), w["kv_fp8"],
        w["kv_scale"], w["block_table"], w["seq_lens"], w["sm_scale"])
    assert_parity(out.float().cpu().numpy().astype(np.float64),
                  lse.cpu().numpy().astype(np.float64), ref_o, ref_l, "f8multi q_len=3")


def test_fp8_bad_block_id_sets_error_bit(lib, oracle_mod):
    w8 = wl.to_fp8(spec("f8bad", 2, 16, 32, [64, 100], seed=4))
    w8 = dict(w8)
    bt = w8["block_table"].copy()
    bt[1, 1] = int(w8["num_blocks"]) + 5
    w8["block_table"] = bt
    out, lse, _ = run_library(w8, check_errors=False)
    m = lib
    assert np.all(np.isfinite(out))
    # request 0 is untouched by the bad entry
    ref_o, ref_l = oracle_ref(oracle_mod, dict(w8, block_table=w8["block_table"][:1],
                                               seq_lens=w8["seq_lens"][:1], q_nope=w8["q_nope"][:1],
                                               q_pe=w8["q_pe"][:1]))
    assert_parity(out[:1], lse[:1], ref_o, ref_l, "f8bad request 0")
    import torch
    t = to_device(w8)
    plan = m.mla_decode_plan(2, 16, w8["seq_lens"], 32, int(w8["max_blocks"]))
    o = torch.empty((2, 16, 512), dtype=torch.bfloat16, device="cuda")
    l = torch.empty((2, 16), dtype=torch.float32, device="cuda")
    m.mla_decode_fp8(plan, t["q_nope"], t["q_pe"], t["kv_fp8"], w8["kv_scale"], t["block_table"],
                     t["seq_lens"], float(w8["sm_scale"]), o, l)
    assert m.mla_check_device_error(plan) == m.MLA_DEVERR_BAD_BLOCK


def test_fp8_kv_scale_is_checked(lib):
    import torch
    m = lib
    w8 = wl.to_fp8(spec("f8arg", 1, 16, 32, [10], seed=2))
    t = to_device(w8)
    plan = m.mla_decode_plan(1, 16, w8["seq_lens"], 32, int(w8["max_blocks"]))
    o = torch.empty((1, 16, 512), dtype=torch.bfloat16, device="cuda")
    l = torch.empty((1, 16), dtype=torch.float32, device="cuda")
    for bad in (0.0, -1.0, float("nan"), float("inf")):
        with pytest.raises(m.MLAError) as e:
            m.mla_decode_fp8(plan, t["q_nope"], t["q_pe"], t["kv_fp8"], bad, t["block_table"],
                             t["seq_lens"], float(w8["sm_scale"]), o, l)
        assert e.value.status == 1
    # a bf16 tensor is not an FP8 cache
    not_fp8 = torch.zeros(tuple(t["kv_fp8"].shape), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(TypeError):
        m.mla_decode_fp8(plan, t["q_nope"], t["q_pe"], not_fp8, 0.1, t["block_table"],
                         t["seq_lens"], 0.07, o, l)
    torch.cuda.synchronize()


def test_fp8_convenience_decode(lib, oracle_mod):
    m = lib
    w8 = wl.to_fp8(spec("f8api", 2, 16, 64, [77, 300], seed=8))
    t = to_device(w8)
    out, lse = m.decode(t["q_nope"], t["q_pe"], t["kv_fp8"], t["block_table"], t["seq_lens"],
                        float(w8["sm_scale"]), seq_lens_host=w8["seq_lens"],
                        kv_scale=w8["kv_scale"])
    ref_o, ref_l = oracle_ref(oracle_mod, w8)
    assert_parity(out.float().cpu().numpy().astype(np.float64),
                  lse.cpu().numpy().astype(np.float64), ref_o, ref_l, "f8api")
