"""The bounded-wait error path on the GPU.

Every wait of the decode roles goes through one bounded routine. A one-warp
kernel waits through it on a barrier that nothing ever completes: the wait
must give up at its limit (about a second) and report MLA_DEVERR_TIMEOUT, by
returning rather than trapping, so that the device stays usable: a decode
issued afterwards still matches the oracle.
"""
import time

import pytest

import mla_workloads as wl
from gpu_helpers import assert_parity, oracle_args, run_library

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


def test_wait_gives_up_and_the_device_stays_usable(lib, oracle_mod):
    t0 = time.perf_counter()
    bits = lib.mla_selftest_wait_timeout()
    elapsed = time.perf_counter() - t0
    assert bits == lib.MLA_DEVERR_TIMEOUT
    assert 0.1 < elapsed < 60.0, elapsed        # the limit is 2e9 SM cycles
    w = wl.generate(wl.WORKLOADS[0])
    out, lse, _ = run_library(w)
    ref_out, ref_lse = oracle_mod.mla_decode(*oracle_args(w))
    assert_parity(out, lse, ref_out, ref_lse, "after the timeout check")
