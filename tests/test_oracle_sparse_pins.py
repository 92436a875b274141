"""Pins of the oracle's sparse (top-k) decode (CPU only).

The sparse decode attends only to the listed tokens of each request. It is
pinned to the bf16 decode, which is pinned on its own:
* listing every token of a request (in any order) gives the full decode;
* listing a subset S gives the full decode of a request whose pages hold
  exactly the rows of S (a cache built by copying those rows), duplicates
  included;
* padding entries (-1, or positions at or past L) change nothing, bit for bit;
* an empty selection gives out = 0 and lse = -inf.
A dropped token, an off-by-one at the length bound or a padding entry taken as
token 0 fails one of them.
"""
import numpy as np

import mla_workloads as wl


def _spec(lens, H=4, bs=16, seed=3):
    return wl.generate(wl.custom_spec("sp", len(lens), H, bs, list(lens), seed=seed))


def _sparse(oracle_mod, w, idx):
    return oracle_mod.mla_decode_sparse(w["q_nope"], w["q_pe"], w["kv_cache"], w["block_table"],
                                        w["seq_lens"], idx, w["sm_scale"])


def _dense(oracle_mod, w):
    return oracle_mod.mla_decode(w["q_nope"], w["q_pe"], w["kv_cache"], w["block_table"],
                                 w["seq_lens"], w["sm_scale"])


def test_all_tokens_listed_is_the_full_decode(oracle_mod):
    w = _spec([7, 50, 33])
    rng = np.random.default_rng(0)
    k = 50
    idx = np.full((3, k), -1, dtype=np.int32)
    for b, L in enumerate(w["seq_lens"]):
        idx[b, :L] = rng.permutation(int(L))
    out, lse = _sparse(oracle_mod, w, idx)
    ref_out, ref_lse = _dense(oracle_mod, w)
    np.testing.assert_allclose(out, ref_out, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def _cache_of_rows(w, b, tokens, bs=16):
    """A one-request workload whose pages hold exactly the rows `tokens` of
    request b of w, in order, with request b's queries."""
    n = len(tokens)
    pages = max(1, -(-n // bs))
    kv = np.full((pages + 1, bs, wl.D), wl.SENTINEL_BF16, dtype=np.uint16)
    for i, t in enumerate(tokens):
        blk = w["block_table"][b, t // w["block_size"]]
        kv[i // bs, i % bs] = w["kv_cache"][blk, t % w["block_size"]]
    return {
        "q_nope": w["q_nope"][b:b + 1], "q_pe": w["q_pe"][b:b + 1], "kv_cache": kv,
        "block_table": np.arange(pages, dtype=np.int32)[None, :],
        "seq_lens": np.array([n], dtype=np.int32), "sm_scale": w["sm_scale"],
    }


def test_subset_is_the_decode_of_those_rows(oracle_mod):
    w = _spec([90, 41])
    idx = np.array([[5, 89, 0, 17, 17, 44, -1, 3],          # 17 listed twice
                    [40, 2, 39, 1, -1, -1, 0, 20]], dtype=np.int32)
    out, lse = _sparse(oracle_mod, w, idx)
    for b in range(2):
        toks = [int(t) for t in idx[b] if 0 <= t < w["seq_lens"][b]]
        ref_out, ref_lse = _dense(oracle_mod, _cache_of_rows(w, b, toks))
        np.testing.assert_allclose(out[b], ref_out[0], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[b], ref_lse[0], rtol=1e-12, atol=1e-12)


def test_padding_entries_change_nothing(oracle_mod):
    w = _spec([30, 30])
    base = np.array([[3, 29, 0, 11], [28, 27, 5, 1]], dtype=np.int32)
    padded = np.array([[3, -1, 29, 30, 0, -7, 11, 31],      # 30, 31: at or past L = 30
                       [-1, 28, 27, 1000, 5, 1, -1, 30]], dtype=np.int32)
    a = _sparse(oracle_mod, w, base)
    b = _sparse(oracle_mod, w, padded)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_token_at_the_length_bound_is_padding(oracle_mod):
    w = _spec([10])
    a = _sparse(oracle_mod, w, np.array([[9, 2]], dtype=np.int32))
    b = _sparse(oracle_mod, w, np.array([[9, 2, 10]], dtype=np.int32))
    np.testing.assert_array_equal(a[0], b[0])
    c = _sparse(oracle_mod, w, np.array([[9]], dtype=np.int32))
    assert not np.allclose(a[0], c[0])   # token 2 does count


def test_empty_selection(oracle_mod):
    w = _spec([12, 0])
    out, lse = _sparse(oracle_mod, w, np.array([[-1, 12, 40], [0, 1, -1]], dtype=np.int32))
    assert np.all(out == 0.0) and np.all(np.isneginf(lse))


def test_generator_selects_distinct_tokens():
    w = wl.with_topk(_spec([5, 300, 0]), 64, seed=4, mixed_padding=True)
    idx = w["topk_indices"]
    for b, L in enumerate(w["seq_lens"]):
        sel = idx[b][(idx[b] >= 0) & (idx[b] < L)]
        assert len(sel) == min(64, int(L)) and len(set(sel.tolist())) == len(sel)


def test_fp8_cache_sparse_is_the_fp8_decode_of_the_list(oracle_mod):
    w8 = wl.to_fp8(_spec([40, 17]))
    rng = np.random.default_rng(5)
    idx = np.full((2, 40), -1, dtype=np.int32)
    for b, L in enumerate(w8["seq_lens"]):
        idx[b, :L] = rng.permutation(int(L))
    out, lse = oracle_mod.mla_decode_sparse(w8["q_nope"], w8["q_pe"], None, w8["block_table"],
                                            w8["seq_lens"], idx, w8["sm_scale"],
                                            kv_fp8=w8["kv_fp8"], kv_scale=w8["kv_scale"])
    ref_out, ref_lse = oracle_mod.mla_decode_fp8(w8["q_nope"], w8["q_pe"], w8["kv_fp8"],
                                                 w8["kv_scale"], w8["block_table"], w8["seq_lens"],
                                                 w8["sm_scale"])
    np.testing.assert_allclose(out, ref_out, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)
