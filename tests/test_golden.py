"""Regression pin of the seeded tiny workload against its stored fixture."""
import hashlib
import json
import os

import numpy as np

import mla_workloads as wl

FIXTURE = os.path.join(os.path.dirname(__file__), "golden", "tiny_b2_h16_oracle.json")


def test_tiny_fixture(oracle_mod):
    with open(FIXTURE) as f:
        g = json.load(f)
    w = wl.generate(wl.WORKLOADS[0])
    for k, h in g["inputs_sha256"].items():
        assert hashlib.sha256(np.ascontiguousarray(w[k]).tobytes()).hexdigest() == h, k
    out, lse = oracle_mod.mla_decode(w["q_nope"], w["q_pe"], w["kv_cache"], w["block_table"],
                                     w["seq_lens"], w["sm_scale"])
    assert np.allclose(lse, np.array(g["lse"]), rtol=0, atol=1e-12)
    assert np.allclose(out.sum(axis=-1), np.array(g["out_row_sums"]), rtol=0, atol=1e-10)
    for key, vals in g["out_samples"].items():
        b, h = map(int, key.split(","))
        assert np.allclose(out[b, h, :8], np.array(vals), rtol=0, atol=1e-12)
    # seq_len 1 request: every head returns the single token's c_kv row.
    row = wl.bf16_bits_to_f32(w["kv_cache"][w["block_table"][0, 0], 0, :512])
    assert np.array_equal(out[0], np.broadcast_to(row.astype(np.float64), (16, 512)))
