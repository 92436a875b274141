"""Pins of the fp64 CPU oracle to facts fixed by the problem, not by itself.

Each test targets a mistake the oracle could plausibly contain:
  - seq_len = 1 returns the token's c_kv row exactly (wrong V columns, wrong
    gather index, a normalisation slip);
  - all-zero queries give the plain mean of V and lse = ln L (wrong log base,
    missing normaliser);
  - identical keys give the mean of V and lse = s + ln L with s from a
    library dot product (dropped q_pe term, missing sm_scale);
  - one dominant key returns that key's V row (sign of the scores, max shift);
  - a two-token case with a closed-form answer in terms of e;
  - the dense single-request case equals scipy's softmax / logsumexp on a
    numpy matrix product (transposed operands, wrong contraction width);
  - physical block permutation leaves the result bit-identical (paging);
  - any split of the tokens merged with the combine equals the unsplit
    result (the split-KV reduction);
  - an independent long-double brute force agrees on tiny shapes;
  - reading one slot past the sequence end is caught by the sentinels.
"""
import math

import numpy as np
import pytest

import mla_workloads as wl

D_C, D_R, D = wl.D_C, wl.D_R, wl.D


def place_rows(rows_per_req, block_size, seed, spare=3):
    """Scatter given per-request token rows (uint16 bf16 [L, 576]) into a
    shuffled paged pool. Returns kv_cache, block_table, seq_lens."""
    rng = np.random.default_rng(seed)
    B = len(rows_per_req)
    lens = np.array([r.shape[0] for r in rows_per_req], dtype=np.int32)
    pages = [(int(L) + block_size - 1) // block_size for L in lens]
    required = sum(pages)
    nb = required + spare
    perm = rng.permutation(nb).astype(np.int32)
    max_blocks = max(1, max(pages) if pages else 1)
    kv = np.full((nb, block_size, D), wl.SENTINEL_BF16, dtype=np.uint16)
    table = np.full((B, max_blocks), perm[-1], dtype=np.int32)
    cur = 0
    for b, rows in enumerate(rows_per_req):
        for p in range(pages[b]):
            blk = perm[cur]
            cur += 1
            table[b, p] = blk
            chunk = rows[p * block_size:(p + 1) * block_size]
            kv[blk, :chunk.shape[0]] = chunk
    return kv, table, lens


def randn_bf16(rng, *shape):
    return wl.f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32))


def f64(bits):
    return wl.bf16_bits_to_f32(bits).astype(np.float64)


def test_seq_len_one_returns_the_row(oracle_mod):
    rng = np.random.default_rng(11)
    H = 5
    rows = [randn_bf16(rng, 1, D), randn_bf16(rng, 1, D)]
    kv, table, lens = place_rows(rows, 16, seed=3)
    qn, qp = randn_bf16(rng, 2, H, D_C), randn_bf16(rng, 2, H, D_R)
    out, lse = oracle_mod.mla_decode(qn, qp, kv, table, lens, 0.07)
    for b in range(2):
        v = f64(rows[b][0, :D_C])
        for h in range(H):
            assert np.array_equal(out[b, h], v)
            s = 0.07 * (np.dot(f64(qn[b, h]), f64(rows[b][0, :D_C]))
                        + np.dot(f64(qp[b, h]), f64(rows[b][0, D_C:])))
            assert abs(lse[b, h] - s) <= 1e-12 * max(1.0, abs(s))


@pytest.mark.parametrize("L,bs", [(1, 16), (7, 16), (33, 32), (200, 64), (129, 128)])
def test_zero_query_is_uniform(oracle_mod, L, bs):
    rng = np.random.default_rng(L)
    rows = randn_bf16(rng, L, D)
    kv, table, lens = place_rows([rows], bs, seed=L + 1)
    qn = np.zeros((1, 3, D_C), np.uint16)
    qp = np.zeros((1, 3, D_R), np.uint16)
    out, lse = oracle_mod.mla_decode(qn, qp, kv, table, lens, 0.5)
    mean = f64(rows[:, :D_C]).mean(axis=0)
    assert np.allclose(out[0], mean[None, :], rtol=0, atol=1e-13)
    assert np.allclose(lse[0], math.log(L), rtol=0, atol=1e-13)


def test_identical_keys_give_mean_of_v(oracle_mod):
    rng = np.random.default_rng(5)
    L, H = 37, 4
    rows = randn_bf16(rng, L, D)
    kpe = randn_bf16(rng, D_R)
    rows[:, D_C:] = kpe[None, :]             # same k_pe for every token
    kv, table, lens = place_rows([rows], 16, seed=9)
    qn = np.zeros((1, H, D_C), np.uint16)     # scores depend on k_pe only
    qp = randn_bf16(rng, 1, H, D_R)
    scale = 1.0 / math.sqrt(192.0)
    out, lse = oracle_mod.mla_decode(qn, qp, kv, table, lens, scale)
    mean = f64(rows[:, :D_C]).mean(axis=0)
    for h in range(H):
        s = scale * float(np.dot(f64(qp[0, h]), f64(kpe)))
        assert np.allclose(out[0, h], mean, rtol=0, atol=1e-12)
        assert abs(lse[0, h] - (s + math.log(L))) <= 1e-12


def test_dominant_key_wins(oracle_mod):
    rng = np.random.default_rng(21)
    L, star = 50, 17
    rows = randn_bf16(rng, L, D)
    rows[:, D_C:] = 0
    rows[star, D_C:] = wl.f32_to_bf16_bits(np.full(D_R, 1.0, np.float32))
    kv, table, lens = place_rows([rows], 32, seed=4)
    qn = np.zeros((1, 2, D_C), np.uint16)
    # q_pe . k_pe(star) = 64 * 1.0 ; with sm_scale = 1 that is a margin of 64 >= 40.
    qp = wl.f32_to_bf16_bits(np.full((1, 2, D_R), 1.0, np.float32))
    out, lse = oracle_mod.mla_decode(qn, qp, kv, table, lens, 1.0)
    for h in range(2):
        assert np.allclose(out[0, h], f64(rows[star, :D_C]), rtol=0, atol=1e-12)
        assert abs(lse[0, h] - 64.0) <= 1e-12
    # Flip the sign of the dominant query: the star token now has the lowest score.
    qp_neg = qp | np.uint16(0x8000)
    out2, _ = oracle_mod.mla_decode(qn, qp_neg, kv, table, lens, 1.0)
    others = np.delete(f64(rows[:, :D_C]), star, axis=0).mean(axis=0)
    assert np.allclose(out2[0, 0], others, rtol=0, atol=1e-12)


def test_two_token_closed_form(oracle_mod):
    # s0 = 0.5 * 0 = 0 and s1 = 0.5 * 2 = 1, so the weights are 1/(1+e), e/(1+e).
    rows = np.zeros((2, D), np.uint16)
    one, two, three = (wl.f32_to_bf16_bits(np.array([v], np.float32))[0] for v in (1, 2, 3))
    rows[0, 1] = one                 # v0 = e_1
    rows[1, 0] = two                 # v1 = 2 e_0 + 3 e_2, and q_nope = e_0 scores it
    rows[1, 2] = three
    kv, table, lens = place_rows([rows], 16, seed=2)
    qn = np.zeros((1, 1, D_C), np.uint16)
    qn[0, 0, 0] = one
    qp = np.zeros((1, 1, D_R), np.uint16)
    out, lse = oracle_mod.mla_decode(qn, qp, kv, table, lens, 0.5)
    e = math.e
    assert abs(lse[0, 0] - math.log(1.0 + e)) < 1e-15
    assert abs(out[0, 0, 0] - 2.0 * e / (1.0 + e)) < 1e-15
    assert abs(out[0, 0, 1] - 1.0 / (1.0 + e)) < 1e-15
    assert abs(out[0, 0, 2] - 3.0 * e / (1.0 + e)) < 1e-15
    assert np.all(out[0, 0, 3:] == 0.0)


def test_dense_case_matches_scipy(oracle_mod):
    special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(8)
    L, H = 70, 6
    rows = randn_bf16(rng, L, D)
    kv, table, lens = place_rows([rows], 16, seed=12)
    qn, qp = randn_bf16(rng, 1, H, D_C), randn_bf16(rng, 1, H, D_R)
    scale = 0.11
    out, lse = oracle_mod.mla_decode(qn, qp, kv, table, lens, scale)
    K = f64(rows)                                   # [L, 576]
    Q = np.concatenate([f64(qn[0]), f64(qp[0])], axis=1)   # [H, 576]
    S = scale * (Q @ K.T)                           # [H, L]
    assert np.allclose(lse[0], special.logsumexp(S, axis=1), rtol=0, atol=1e-12)
    assert np.allclose(out[0], special.softmax(S, axis=1) @ K[:, :D_C], rtol=0, atol=1e-12)


def test_block_permutation_is_bit_invariant(oracle_mod):
    w = wl.generate(wl.custom_spec("perm", B=3, H=4, block_size=16, seq_lens=[40, 1, 77],
                                   seed=31))
    w2 = wl.permute_blocks(w, seed=99)
    assert not np.array_equal(w["block_table"], w2["block_table"])
    args = ("q_nope", "q_pe", "kv_cache", "block_table", "seq_lens")
    o1, l1 = oracle_mod.mla_decode(*(w[k] for k in args), w["sm_scale"])
    o2, l2 = oracle_mod.mla_decode(*(w2[k] for k in args), w2["sm_scale"])
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("cuts", [[1], [64], [5, 6, 100], [13, 50, 51, 127]])
def test_split_then_combine_equals_unsplit(oracle_mod, cuts):
    w = wl.generate(wl.custom_spec("split", B=2, H=3, block_size=32, seq_lens=[128, 9],
                                   seed=7, peaky_fraction=0.05))
    args = [w[k] for k in ("q_nope", "q_pe", "kv_cache", "block_table", "seq_lens")]
    full_o, full_l = oracle_mod.mla_decode(*args, w["sm_scale"])
    L = int(w["seq_lens"][0])
    bounds = [0] + [c for c in cuts if c < L] + [L]
    for h in range(3):
        parts = [oracle_mod.mla_partial(*args, w["sm_scale"], 0, h, a, b)
                 for a, b in zip(bounds[:-1], bounds[1:])]
        o, l = oracle_mod.mla_combine(np.stack([p[0] for p in parts]),
                                      np.array([p[1] for p in parts]))
        assert np.allclose(o, full_o[0, h], rtol=0, atol=1e-12)
        assert abs(l - full_l[0, h]) <= 1e-12


def test_combine_ignores_empty_partials(oracle_mod):
    rng = np.random.default_rng(0)
    o_parts = rng.standard_normal((3, D_C))
    lse_parts = np.array([0.3, -np.inf, 1.2])
    o, l = oracle_mod.mla_combine(o_parts, lse_parts)
    o2, l2 = oracle_mod.mla_combine(o_parts[[0, 2]], lse_parts[[0, 2]])
    assert np.array_equal(o, o2) and l == l2
    o3, l3 = oracle_mod.mla_combine(o_parts[:1], np.array([-np.inf]))
    assert l3 == -np.inf and np.all(o3 == 0.0)


@pytest.mark.parametrize("bs,lens,H", [(16, [1, 16, 17], 2), (32, [40, 0, 5], 3),
                                       (64, [130], 1), (128, [3, 255], 2)])
def test_bruteforce_agrees(oracle_mod, bs, lens, H):
    w = wl.generate(wl.custom_spec("bf", B=len(lens), H=H, block_size=bs, seq_lens=lens,
                                   seed=sum(lens) + bs))
    args = [w[k] for k in ("q_nope", "q_pe", "kv_cache", "block_table", "seq_lens")]
    o1, l1 = oracle_mod.mla_decode(*args, w["sm_scale"])
    o2, l2 = oracle_mod.mla_decode_bruteforce(*args, w["sm_scale"])
    assert np.allclose(o1, o2, rtol=0, atol=1e-12)
    finite = np.isfinite(l2)
    assert np.array_equal(finite, np.isfinite(l1))
    assert np.allclose(l1[finite], l2[finite], rtol=0, atol=1e-12)


def test_empty_sequence(oracle_mod):
    w = wl.generate(wl.custom_spec("empty", B=2, H=2, block_size=16, seq_lens=[0, 3], seed=4))
    args = [w[k] for k in ("q_nope", "q_pe", "kv_cache", "block_table", "seq_lens")]
    o, l = oracle_mod.mla_decode(*args, w["sm_scale"])
    assert np.all(o[0] == 0.0) and np.all(l[0] == -np.inf)
    assert np.all(np.isfinite(l[1]))


def test_rows_api_matches_full(oracle_mod):
    w = wl.generate(wl.custom_spec("rows", B=3, H=5, block_size=32, seq_lens=[70, 2, 33],
                                   seed=6))
    args = [w[k] for k in ("q_nope", "q_pe", "kv_cache", "block_table", "seq_lens")]
    o, l = oracle_mod.mla_decode(*args, w["sm_scale"])
    rb, rh = np.array([2, 0, 1, 2]), np.array([4, 0, 3, 1])
    orow, lrow = oracle_mod.mla_decode_rows(*args, w["sm_scale"], rb, rh)
    assert np.array_equal(orow, o[rb, rh]) and np.array_equal(lrow, l[rb, rh])


def test_heads_and_requests_are_independent(oracle_mod):
    w = wl.generate(wl.custom_spec("indep", B=2, H=4, block_size=16, seq_lens=[20, 31],
                                   seed=13))
    keys = ("q_nope", "q_pe", "kv_cache", "block_table", "seq_lens")
    o1, l1 = oracle_mod.mla_decode(*(w[k] for k in keys), w["sm_scale"])
    w2 = dict(w)
    qn = w["q_nope"].copy()
    qn[1, 2] = qn[1, 2] ^ np.uint16(0x8000)          # flip one head of request 1
    w2["q_nope"] = qn
    o2, l2 = oracle_mod.mla_decode(*(w2[k] for k in keys), w2["sm_scale"])
    changed = np.zeros((2, 4), bool)
    changed[1, 2] = True
    assert np.array_equal(o1[~changed], o2[~changed]) and np.array_equal(l1[~changed], l2[~changed])
    assert not np.allclose(o1[1, 2], o2[1, 2])


def test_reading_past_the_end_is_caught_by_sentinels(oracle_mod):
    # Plant the mistake in the oracle's inputs: claim one token more than the
    # request has. The extra row is a +-9984 sentinel, and the result moves far
    # outside the parity tolerance |d| <= 2e-2 + 2e-2 |ref|.
    w = wl.generate(wl.custom_spec("sent", B=1, H=8, block_size=32, seq_lens=[45], seed=17))
    keys = ("q_nope", "q_pe", "kv_cache", "block_table")
    o1, _ = oracle_mod.mla_decode(*(w[k] for k in keys), w["seq_lens"], w["sm_scale"])
    o2, _ = oracle_mod.mla_decode(*(w[k] for k in keys), w["seq_lens"] + 1, w["sm_scale"])
    # A sentinel row scores about +-1.7e4 per head: heads that score it
    # positively are dominated by it, the others give it weight exp(-1.7e4) = 0.
    # So the stray read is caught by some head of the request (each head
    # misses with probability 1/2 independently), not by every head.
    excess = (np.abs(o2 - o1) - (2e-2 + 2e-2 * np.abs(o1))).max(axis=-1)[0]
    caught = excess > 0
    assert caught.any()
    assert np.all(np.abs(o2[0, caught]).max(axis=-1) > 9000.0)


def test_bad_block_id_is_reported(oracle_mod):
    w = wl.generate(wl.custom_spec("bad", B=1, H=1, block_size=16, seq_lens=[20], seed=1))
    table = w["block_table"].copy()
    table[0, 1] = w["num_blocks"]                   # out of range
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.mla_decode(w["q_nope"], w["q_pe"], w["kv_cache"], table, w["seq_lens"],
                              w["sm_scale"])
