"""Write the regression fixture of the tiny decode workload.

Calls only the oracle package and the seeded input generator. Run from the
repository root:  python tests/golden/make_golden.py
"""
import hashlib
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import mla_workloads as wl  # noqa: E402
import oracle  # noqa: E402

PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_b2_h16_oracle.json")
SAMPLE_ROWS = [(0, 0), (0, 15), (1, 3), (1, 15)]


def digest(a: np.ndarray) -> str:
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


def make():
    w = wl.generate(wl.WORKLOADS[0])
    out, lse = oracle.mla_decode(w["q_nope"], w["q_pe"], w["kv_cache"], w["block_table"],
                                 w["seq_lens"], w["sm_scale"])
    return {
        "workload": w["name"],
        "source": "written by tests/golden/make_golden.py from the oracle package; the pages "
                  "print no worked example for MLA decode",
        "inputs_sha256": {k: digest(w[k]) for k in ("q_nope", "q_pe", "kv_cache",
                                                   "block_table", "seq_lens")},
        "lse": [[float(x) for x in row] for row in lse],
        "out_row_sums": [[float(x) for x in row] for row in out.sum(axis=-1)],
        "out_samples": {f"{b},{h}": [float(x) for x in out[b, h, :8]] for b, h in SAMPLE_ROWS},
    }


if __name__ == "__main__":
    with open(PATH, "w") as f:
        json.dump(make(), f, indent=1)
    print("wrote", PATH)
