"""Pins of the oracle's FP8-cache decode (CPU only).

The FP8 path adds two things to the pinned bf16 decode: the E4M3 byte
decoding and one per-tensor scale applied to every cached element. Each is
pinned to something outside the oracle's own code:

* the 256 E4M3 codes against torch's float8_e4m3fn widening (an independent
  library implementation of the OCP format) and against landmark values the
  format fixes (largest finite 448, smallest normal 2^-6, smallest subnormal
  2^-9, no infinities, two NaN codes);
* the scale through the linearity of attention in the cache: with every
  element multiplied by s, the scores are those of sm_scale * s and the output
  is s times the unscaled output. So the FP8 decode must equal s times the
  bf16 decode (pinned elsewhere) of the decoded values under sm_scale * s. A
  scale dropped from K or from V, or applied twice, fails it;
* closed forms: a one-token sequence returns kv_scale * e4m3(row[:512]);
  identical rows return that row; the block placement does not matter.
"""
import numpy as np
import pytest

import mla_workloads as wl


def _tiny(name="fp8pin", B=3, H=4, bs=16, lens=(1, 37, 70), seed=5, peaky=0.0):
    return wl.generate(wl.custom_spec(name, B, H, bs, list(lens), seed=seed,
                                      peaky_fraction=peaky))


def test_e4m3_decode_matches_torch_float8(oracle_mod):
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle_mod.e4m3_decode(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert np.array_equal(np.signbit(ours[ok]), np.signbit(ref[ok]))


def test_e4m3_format_landmarks(oracle_mod):
    cases = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
             0x38: 1.0, 0x3F: 1.875, 0x40: 2.0, 0x7E: 448.0, 0xC0: -2.0, 0xFE: -448.0,
             0x77: 240.0, 0x0F: 1.875 * 2.0 ** -6}
    codes = np.array(list(cases), dtype=np.uint8)
    got = oracle_mod.e4m3_decode(codes)
    assert got.tolist() == list(cases.values())
    neg0 = oracle_mod.e4m3_decode(np.array([0x80], dtype=np.uint8))[0]
    assert neg0 == 0.0 and np.signbit(neg0)
    nan = oracle_mod.e4m3_decode(np.array([0x7F, 0xFF], dtype=np.uint8))
    assert np.isnan(nan).all()
    # no infinities: every other code is finite and at most 448 in magnitude
    allv = oracle_mod.e4m3_decode(np.arange(256, dtype=np.uint8))
    fin = allv[~np.isnan(allv)]
    assert fin.size == 254 and np.abs(fin).max() == 448.0


def _decoded_as_bf16(oracle_mod, w8):
    """The decoded E4M3 values as a bf16 cache (exact: 4 significant bits and
    exponents -9..8 all fit bf16)."""
    vals = oracle_mod.e4m3_decode(w8["kv_fp8"]).astype(np.float32)
    bits = wl.f32_to_bf16_bits(vals)
    assert np.array_equal(wl.bf16_bits_to_f32(bits), vals)
    return bits


@pytest.mark.parametrize("scale", [0.1, 0.25, 3.0])
def test_fp8_decode_is_scaled_bf16_decode(oracle_mod, scale):
    w = _tiny(peaky=0.05)
    w8 = wl.to_fp8(w, kv_scale=scale)
    out8, lse8 = oracle_mod.mla_decode_fp8(w8["q_nope"], w8["q_pe"], w8["kv_fp8"], scale,
                                           w8["block_table"], w8["seq_lens"], w8["sm_scale"])
    ref_out, ref_lse = oracle_mod.mla_decode(w8["q_nope"], w8["q_pe"], _decoded_as_bf16(oracle_mod, w8),
                                             w8["block_table"], w8["seq_lens"],
                                             w8["sm_scale"] * scale)
    np.testing.assert_allclose(out8, scale * ref_out, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse8, ref_lse, rtol=1e-12, atol=1e-12)


def test_fp8_single_token_returns_scaled_row(oracle_mod):
    w = _tiny(B=2, lens=(1, 1))
    w8 = wl.to_fp8(w, kv_scale=0.1)
    out, lse = oracle_mod.mla_decode_fp8(w8["q_nope"], w8["q_pe"], w8["kv_fp8"], 0.1,
                                         w8["block_table"], w8["seq_lens"], w8["sm_scale"])
    for b in range(2):
        row = w8["kv_fp8"][w8["block_table"][b, 0], 0, :512]
        want = 0.1 * oracle_mod.e4m3_decode(row)
        for h in range(w8["H"]):
            np.testing.assert_allclose(out[b, h], want, rtol=1e-14, atol=0)


def test_fp8_identical_rows_return_the_row(oracle_mod):
    w = _tiny(B=1, lens=(53,))
    w8 = wl.to_fp8(w, kv_scale=0.1)
    kv = w8["kv_fp8"].copy()
    src = kv[w8["block_table"][0, 0], 0].copy()
    for t in range(53):
        kv[w8["block_table"][0, t // 16], t % 16] = src
    out, lse = oracle_mod.mla_decode_fp8(w8["q_nope"], w8["q_pe"], kv, 0.1, w8["block_table"],
                                         w8["seq_lens"], w8["sm_scale"])
    want = 0.1 * oracle_mod.e4m3_decode(src[:512])
    np.testing.assert_allclose(out[0], np.broadcast_to(want, out[0].shape), rtol=1e-12, atol=1e-14)


def test_fp8_block_permutation_invariance(oracle_mod):
    w8 = wl.to_fp8(_tiny(lens=(5, 64, 99)), kv_scale=0.1)
    p8 = wl.permute_blocks(w8, seed=77)
    a = oracle_mod.mla_decode_fp8(w8["q_nope"], w8["q_pe"], w8["kv_fp8"], 0.1, w8["block_table"],
                                  w8["seq_lens"], w8["sm_scale"])
    b = oracle_mod.mla_decode_fp8(p8["q_nope"], p8["q_pe"], p8["kv_fp8"], 0.1, p8["block_table"],
                                  p8["seq_lens"], p8["sm_scale"])
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_fp8_multi_token_is_scaled_bf16_multi_token(oracle_mod):
    w = _tiny(B=2, H=3, lens=(9, 40))
    rng = np.random.default_rng(3)
    q_len = 3
    qn = wl.f32_to_bf16_bits(rng.standard_normal((2, q_len, 3, 512), dtype=np.float32))
    qp = wl.f32_to_bf16_bits(rng.standard_normal((2, q_len, 3, 64), dtype=np.float32))
    w8 = wl.to_fp8(w, kv_scale=0.1)
    out8, lse8 = oracle_mod.mla_decode_fp8(qn, qp, w8["kv_fp8"], 0.1, w8["block_table"],
                                           w8["seq_lens"], w8["sm_scale"])
    ref_out, ref_lse = oracle_mod.mla_decode_multi(qn, qp, _decoded_as_bf16(oracle_mod, w8),
                                                   w8["block_table"], w8["seq_lens"],
                                                   w8["sm_scale"] * 0.1)
    assert out8.shape == (2, q_len, 3, 512) and lse8.shape == (2, q_len, 3)
    np.testing.assert_allclose(out8, 0.1 * ref_out, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse8, ref_lse, rtol=1e-12, atol=1e-12)


def test_fp8_workload_sentinels_are_largest_codes():
    w = _tiny(lens=(5, 17, 33))
    w8 = wl.to_fp8(w, kv_scale=0.1)
    spare = w8["spare_blocks"]
    mags = w8["kv_fp8"][spare] & 0x7F
    assert (mags == 0x7E).all()          # +-448: the sentinel saturates
    assert not np.isin(w8["kv_fp8"], [0x7F, 0xFF]).any()
