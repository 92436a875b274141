"""The N > 1 host logic of bench.py, run as two gloo ranks on the CPU.

The decode needs no collective, so several GPUs run independent replicas; the
only cross-rank steps are the barrier around the timed region and the max of
the per-rank times. The reference arm runs on rank 0 alone while the other
ranks exit without work.
"""
import multiprocessing as mp
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    try:
        import bench
        dist = bench.init_dist(world, "gloo")
        bench.barrier(dist)
        # Each rank reports its own step time; every rank must see the max.
        got = bench.max_over_ranks(10.0 + 3.0 * rank, dist)
        bench.barrier(dist)
        dist.destroy_process_group()
        q.put((rank, "max", got))
    except Exception as e:  # pragma: no cover - reported through the queue
        q.put((rank, "error", repr(e)))


def _reference_rank(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    try:
        import argparse
        import bench
        args = argparse.Namespace(steps=1, warmup=3, config="tiny_b2_h16", kv="bf16", q_len=1,
                                  graph=False)
        res = bench.bench_reference(args, world, rank, rank)
        q.put((rank, "ref", None if res is None else (res["impl"], res["n_gpus"], res["value"] > 0)))
    except Exception as e:  # pragma: no cover
        q.put((rank, "error", repr(e)))


def _run(target, world=2):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=target, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = {}
    for _ in range(world):
        rank, kind, val = q.get(timeout=240)
        assert kind != "error", f"rank {rank}: {val}"
        out[rank] = val
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return out


def test_max_over_two_gloo_ranks():
    out = _run(_rank_main)
    assert out == {0: 13.0, 1: 13.0}


def test_reference_arm_runs_on_rank_zero_only():
    pytest.importorskip("torch")
    out = _run(_reference_rank)
    assert out[1] is None
    assert out[0] == ("reference", 2, True)
