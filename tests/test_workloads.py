"""The seeded input generator: layout, sentinels and determinism."""
import numpy as np
import pytest

import mla_workloads as wl


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-9, -2.5, 1e4], np.float32)
    bits = wl.f32_to_bf16_bits(x)
    back = wl.bf16_bits_to_f32(bits)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: even mantissa (1.0) wins.
    assert back.tolist() == [1.0, 1.0, 1.0 + 2**-7, -2.5, 9984.0]
    assert bits[-1] == wl.SENTINEL_BF16


@pytest.mark.parametrize("idx", [0, 1])
def test_layout_and_sentinels(idx):
    w = wl.generate(wl.WORKLOADS[idx])
    bs, nb = w["block_size"], w["num_blocks"]
    seq, table, kv = w["seq_lens"], w["block_table"], w["kv_cache"]
    spare = set(w["spare_blocks"].tolist())
    used = []
    for b in range(w["B"]):
        n = (int(seq[b]) + bs - 1) // bs
        used += table[b, :n].tolist()
        assert all(int(x) in spare for x in table[b, n:])
        if seq[b] % bs:
            tail = kv[table[b, n - 1], seq[b] % bs:]
            assert np.all((tail & 0x7FFF) == wl.SENTINEL_BF16)
    assert len(used) == len(set(used)) and not (set(used) & spare)
    assert set(used) | spare == set(range(nb))
    for s in list(spare)[:3]:
        assert np.all((kv[s] & 0x7FFF) == wl.SENTINEL_BF16)
    # Valid rows look like bf16(N(0,1)) and never hold a sentinel magnitude.
    b0 = int(np.argmax(seq))
    v = wl.bf16_bits_to_f32(kv[table[b0, 0]])
    assert abs(float(v.mean())) < 0.1 and 0.9 < float(v.std()) < 1.1


def test_determinism_and_seed_dependence():
    s = wl.custom_spec("d", B=2, H=2, block_size=16, seq_lens=[5, 40], seed=3)
    a, b = wl.generate(s), wl.generate(s)
    for k in ("kv_cache", "q_nope", "q_pe", "block_table"):
        assert np.array_equal(a[k], b[k])
    c = wl.generate(wl.custom_spec("d", B=2, H=2, block_size=16, seq_lens=[5, 40], seed=4))
    assert not np.array_equal(a["kv_cache"], c["kv_cache"])


def test_config_shapes():
    names = [w.name for w in wl.WORKLOADS]
    assert names == ["tiny_b2_h16", "v2lite_b64_h16", "r1_b128_h128", "r1_b512_h128",
                     "long_b4_h128"]
    tiny = wl.generate(wl.WORKLOADS[0])
    assert tiny["seq_lens"].tolist() == [1, 256] and tiny["num_blocks"] == 13
    assert tiny["q_nope"].shape == (2, 16, 512) and tiny["kv_cache"].shape == (13, 32, 576)


def test_peaky_rows_scaled_by_eight():
    s = wl.custom_spec("p", B=1, H=1, block_size=16, seq_lens=[3000], seed=9,
                       peaky_fraction=0.01)
    s0 = wl.custom_spec("p", B=1, H=1, block_size=16, seq_lens=[3000], seed=9)
    w = wl.generate(s)
    big = np.abs(wl.bf16_bits_to_f32(w["kv_cache"])).max(axis=-1)
    valid = np.zeros_like(big, dtype=bool)
    for p in range(3000 // 16 + 1):
        n = min(16, 3000 - 16 * p)
        if n > 0:
            valid[w["block_table"][0, p], :n] = True
    frac = float((big[valid] > 20.0).mean())
    assert 0.003 < frac < 0.03
    assert s0.peaky_fraction == 0.0


def test_permute_blocks_keeps_logical_rows():
    w = wl.generate(wl.custom_spec("perm", B=2, H=1, block_size=16, seq_lens=[30, 7], seed=2))
    w2 = wl.permute_blocks(w, seed=5)
    for b in range(2):
        for p in range(2):
            assert np.array_equal(w["kv_cache"][w["block_table"][b, p]],
                                  w2["kv_cache"][w2["block_table"][b, p]])


def test_expected_counts():
    w = wl.generate(wl.WORKLOADS[0])
    c = wl.expected_counts(w)
    assert c["tokens"] == 257
    assert c["kv_bytes"] == 257 * 1152
    assert c["flops"] == 257 * 16 * (2 * 576 + 2 * 512)


def test_sparse_counts_match_dense_counts_on_full_lists():
    """With every token of every request listed once, the sparse accounting
    has the dense one's KV bytes, flops and token count; it differs only in
    the index bytes (4 per list entry) and the table bytes (4 per listed
    token instead of 4 per page)."""
    w = wl.generate(wl.custom_spec("cnt", 3, 16, 32, [5, 70, 0], seed=2))
    topk = 70
    idx = np.full((3, topk), -1, dtype=np.int32)
    for b, L in enumerate(w["seq_lens"]):
        idx[b, :L] = np.arange(L)
    ws = dict(w, topk_indices=idx)
    dense, sparse = wl.expected_counts(w), wl.sparse_counts(ws)
    assert sparse["tokens"] == dense["tokens"] == 75
    assert sparse["kv_bytes"] == dense["kv_bytes"] and sparse["flops"] == dense["flops"]
    pages = sum(-(-int(L) // 32) for L in w["seq_lens"])
    assert sparse["bytes"] - dense["bytes"] == 4 * idx.size + 4 * 75 - 4 * pages
    # padding and repeats: a repeat counts again, padding not at all
    idx2 = np.array([[0, 0, -1, 5, 4], [69, 70, 1, 1, 1], [0, -1, -1, -1, -1]], dtype=np.int32)
    assert wl.sparse_counts(dict(w, topk_indices=idx2))["tokens"] == 3 + 4 + 0
    assert wl.sparse_counts(wl.to_fp8(ws))["kv_bytes"] == 75 * 576
