"""Pins of the oracle's multi-token (speculative) decode.

Reading taken where the pages only name speculative decoding: a request of
length L holds q_len new tokens as its last q_len tokens, and query token j
attends causally to tokens t < L - q_len + 1 + j. The pins tie the
multi-token routine to the single-token decode, whose own pins are in
test_oracle_pins.py, and check the causal boundary from both sides:
  - q_len = 1 is exactly the single-token decode;
  - every row (b, j, h) equals the single-token decode of query row j on the
    request truncated to L - q_len + 1 + j tokens (an off-by-one in the causal
    length, or a [q_len, H] / [H, q_len] layout slip, fails it);
  - changing the first token hidden from row j leaves row j bit-identical
    and changes row j + 1;
  - an empty request gives out = 0 and lse = -inf for every row.
"""
import numpy as np
import pytest

import mla_workloads as wl


def multi_workload(B, q_len, H, bs, lens, seed):
    """A generated workload with q_len * H query rows per request, viewed as
    q [B, q_len, H, ...] (the generator's draws, reshaped)."""
    w = wl.generate(wl.custom_spec("multi", B=B, H=q_len * H, block_size=bs, seq_lens=lens,
                                   seed=seed))
    w = dict(w)
    w["q_nope4"] = w["q_nope"].reshape(B, q_len, H, wl.D_C)
    w["q_pe4"] = w["q_pe"].reshape(B, q_len, H, wl.D_R)
    return w


def test_single_token_is_the_plain_decode(oracle_mod):
    w = multi_workload(3, 1, 8, 32, [1, 77, 300], seed=1)
    o1, l1 = oracle_mod.mla_decode_multi(w["q_nope4"], w["q_pe4"], w["kv_cache"],
                                         w["block_table"], w["seq_lens"], w["sm_scale"])
    o0, l0 = oracle_mod.mla_decode(w["q_nope"], w["q_pe"], w["kv_cache"], w["block_table"],
                                   w["seq_lens"], w["sm_scale"])
    assert np.array_equal(o1[:, 0], o0) and np.array_equal(l1[:, 0], l0)


@pytest.mark.parametrize("q_len", [2, 3, 5])
def test_each_row_is_the_truncated_single_token_decode(oracle_mod, q_len):
    H = 4
    lens = [q_len, 40, 129, 300]
    w = multi_workload(4, q_len, H, 32, lens, seed=q_len)
    out, lse = oracle_mod.mla_decode_multi(w["q_nope4"], w["q_pe4"], w["kv_cache"],
                                           w["block_table"], w["seq_lens"], w["sm_scale"])
    B = len(lens)
    for j in range(q_len):
        lens_j = np.array([L - q_len + 1 + j for L in lens], dtype=np.int32)
        rb = np.repeat(np.arange(B), H)
        rh = np.tile(np.arange(H), B) + j * H          # row j * H + h of the request
        ro, rl = oracle_mod.mla_decode_rows(w["q_nope"], w["q_pe"], w["kv_cache"],
                                            w["block_table"], lens_j, w["sm_scale"], rb, rh)
        assert np.array_equal(out[:, j].reshape(-1, wl.D_C), ro)
        assert np.array_equal(lse[:, j].reshape(-1), rl)


def test_causal_boundary(oracle_mod):
    q_len, H, L = 4, 2, 100
    w = multi_workload(1, q_len, H, 16, [L], seed=9)
    out, lse = oracle_mod.mla_decode_multi(w["q_nope4"], w["q_pe4"], w["kv_cache"],
                                           w["block_table"], w["seq_lens"], w["sm_scale"])
    for j in range(q_len - 1):
        t = L - q_len + 1 + j              # first token hidden from row j, seen by row j + 1
        kv = w["kv_cache"].copy()
        blk, slot = w["block_table"][0, t // 16], t % 16
        kv[blk, slot] = wl.f32_to_bf16_bits(wl.bf16_bits_to_f32(kv[blk, slot]) * np.float32(3.0))
        o2, l2 = oracle_mod.mla_decode_multi(w["q_nope4"], w["q_pe4"], kv, w["block_table"],
                                             w["seq_lens"], w["sm_scale"])
        assert np.array_equal(o2[0, : j + 1], out[0, : j + 1])
        assert np.array_equal(l2[0, : j + 1], lse[0, : j + 1])
        assert not np.allclose(o2[0, j + 1], out[0, j + 1])


def test_empty_request_rows(oracle_mod):
    w = multi_workload(2, 3, 2, 32, [0, 5], seed=4)
    out, lse = oracle_mod.mla_decode_multi(w["q_nope4"], w["q_pe4"], w["kv_cache"],
                                           w["block_table"], w["seq_lens"], w["sm_scale"])
    assert np.all(out[0] == 0) and np.all(lse[0] == -np.inf)
    assert np.all(np.isfinite(out[1])) and np.all(np.isfinite(lse[1]))


def test_too_short_request_is_refused(oracle_mod):
    w = multi_workload(1, 3, 2, 32, [2], seed=4)
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.mla_decode_multi(w["q_nope4"], w["q_pe4"], w["kv_cache"], w["block_table"],
                                    w["seq_lens"], w["sm_scale"])
