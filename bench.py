"""Benchmark of the paged MLA decode (one JSON line on stdout, rank 0).

Default workload: the high-concurrency decode, B=512 requests, H=128 heads,
lengths 1024 + U{0..2048}, block size 32, a 35,265-block (~1.3 GB) bf16 latent
cache (seeded synthetic data; the pages' kernel-only microbenchmark shape at
bs=512, see "[Kernel] Flashinfer MLA (trtllm-gen) decode kernel integration",
Kernel-only microbenchmark). A step is one ``mla_decode`` call (decode kernel,
plus the combine kernel when the plan splits a request) with inputs resident
in HBM; the cache alone is ten times the 129 MB L2, so no flush is needed
between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config NAME] [--kv bf16|fp8]

``--kv fp8`` runs the same workload over an FP8 (E4M3, per-tensor scale)
cache through ``mla_decode_fp8`` (576 bytes per cached token). ``--q-len N``
gives every request N query tokens (speculative decoding, causal within the
request's last N tokens; at 128 heads that is N head groups of 128 rows).
``--graph`` captures one step in a CUDA graph, with a plan built for length
bounds, and times its replays.

``--config sparse_r1_b64_h128`` runs the sparse (top-k) decode instead: B=64,
H=128, lengths 8192 + U{0..8192}, each request attending to 2048 listed tokens
(``mla_decode_sparse``: gather kernel, then the decode kernel).

``--impl reference`` times the fp64 CPU oracle on a bounded sample of the
same workload on the host cores (the slow baseline). Under torchrun (N > 1)
every rank runs its own replica of the workload (the decode needs no
collective); the timing is max-reduced over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import mla_workloads as wl  # noqa: E402

METRIC = "MLA decode µs/call + KV-read HBM GB/s at B=512,H=128 vs roofline fraction"
UNIT = "us/call"
DEFAULT_CONFIG = "r1_b512_h128"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# The sources the paged decode kernel is compiled from (the recorded DRAM
# traffic is used only while they are unchanged).
DECODE_SRCS = [os.path.join(ROOT, "paged_mla_decode_05_gb300", "csrc", f)
               for f in ("mla_decode_kernel.cuh", "mla_decode_sm103.cu", "ptx_sm103.cuh",
                         "mla_internal.h")]
TRAFFIC_FILES = {"bf16": os.path.join(ROOT, "profiles", "decode_r1_b512_h128_traffic.txt"),
                 "fp8": os.path.join(ROOT, "profiles", "decode_r1_b512_h128_fp8_traffic.txt")}
FP8_OVER_BF16 = 2.0   # nominal dense fp8 / bf16 tensor throughput (4.5 / 2.25 PFLOP/s)
L2_BYTES = 129 * 1024 * 1024      # GB300 L2
FLUSH_BYTES = 512 * 1024 * 1024   # written between steps when the cache is near the L2 size


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ----------------------------------------------------------------- distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(value: float, dist, device=None) -> float:
    """Max of a float over all ranks (identity without a process group)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ---------------------------------------------------------------- measurements

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_digest() -> str:
    h = hashlib.sha256()
    for path in DECODE_SRCS:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(config: str, kv: str):
    """DRAM bytes per decode launch of the default workload from the committed
    ncu summary, if it was taken on the current kernel source (else None)."""
    path = TRAFFIC_FILES[kv]
    if config != DEFAULT_CONFIG or not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line:
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("kernel_source_sha256_16") != source_digest():
        return None
    try:
        return float(vals["dram_bytes_per_launch_full_workload"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self._t.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def spec_of(name: str):
    return wl.SPARSE_WORKLOADS[name] if is_sparse(name) else wl.WORKLOADS_BY_NAME[name]


def is_sparse(name: str) -> bool:
    return name in wl.SPARSE_WORKLOADS


def load_workload(name: str, kv: str, q_len: int = 1):
    """The seeded workload, with its cache converted to E4M3 for kv == "fp8";
    a sparse workload also gets its top-k lists (seeded by the spec's seed);
    q_len > 1 gives each request q_len query tokens (speculative decoding)."""
    spec = spec_of(name)
    if q_len > 1:
        if is_sparse(name):
            raise SystemExit("--q-len applies to the dense workloads only")
        w = wl.multi_token(spec, q_len)
    else:
        w = wl.generate(spec)
    if is_sparse(name):
        w = wl.with_topk(w, wl.SPARSE_TOPK, seed=spec.seed)
    return wl.to_fp8(w) if kv == "fp8" else w


def counts_of(w):
    return wl.sparse_counts(w) if "topk_indices" in w else wl.expected_counts(w)


def request_work(w):
    """Tokens each request attends to: its length, or its valid list entries."""
    seq = np.asarray(w["seq_lens"], dtype=np.int64)
    if "topk_indices" not in w:
        return seq
    idx = np.asarray(w["topk_indices"], dtype=np.int64)
    return ((idx >= 0) & (idx < seq[:, None])).sum(axis=1)


def cache_of(w):
    return w["kv_fp8"] if "kv_fp8" in w else w["kv_cache"]


def workload_config(spec, w, counts, world, graph=False):
    """The config block both arms report for a workload (identical keys)."""
    cache_bytes = int(cache_of(w).nbytes)
    fp8 = "kv_fp8" in w
    q_len = int(w.get("q_len", 1))
    extra = {}
    if q_len > 1:
        extra = {"q_len": q_len, "heads": int(w["heads"]),
                 "query_rows_per_request": int(w["H"]),
                 "causal": "query token j sees the first L - q_len + 1 + j tokens"}
    if graph:
        extra["launch"] = ("CUDA graph replay of one captured step (plan built for length "
                           "bounds; the kernels read the lengths on the device)")
    sparse = {"topk": int(w["topk_indices"].shape[1]),
              "selection": "min(topk, L) distinct positions per request, uniform"} \
        if "topk_indices" in w else {}
    name = spec.name + (f"_q{q_len}" if q_len > 1 else "") + ("_fp8" if fp8 else "")
    return {"workload": name, "B": int(w["B"]), "H": int(w.get("heads", w["H"])),
            **sparse, **extra,
            "kv_cache": (f"fp8 e4m3, per-tensor scale {w['kv_scale']}" if fp8 else "bf16"),
            "block_size": int(w["block_size"]),
            "seq_lens": "1024+U{0..2048}" if spec.name.startswith("r1_") else spec.description,
            "tokens": counts["tokens"], "num_blocks": int(w["num_blocks"]),
            "cache_bytes": cache_bytes,
            "l2": (f"L2 flushed before every step ({FLUSH_BYTES >> 20} MB write, untimed)"
                   if cache_bytes < 4 * L2_BYTES else
                   f"inputs larger than L2 (cache {cache_bytes / L2_BYTES:.0f}x the 129 MB L2); no flush"),
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


# -------------------------------------------------------------- our GPU path

def bench_ours(args, world, rank, local):
    import torch
    dist = init_dist(world, "nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import paged_mla_decode_05_gb300 as m
    from paged_mla_decode_05_gb300 import build as _b
    _b.build()

    spec = spec_of(args.config)
    t0 = time.time()
    w = load_workload(args.config, args.kv, args.q_len)
    fp8 = args.kv == "fp8"
    sparse = is_sparse(args.config)
    q_len = int(w.get("q_len", 1))
    heads = int(w.get("heads", w["H"]))
    log(f"[bench] generated {spec.name} ({args.kv} cache) in {time.time() - t0:.1f}s")
    counts = counts_of(w)
    B, H, bs = w["B"], w["H"], w["block_size"]

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    q_nope, q_pe = bf16(w["q_nope"]), bf16(w["q_pe"])
    kv = torch.from_numpy(w["kv_fp8"]).to(dev) if fp8 else bf16(w["kv_cache"])
    table = torch.from_numpy(w["block_table"]).to(dev)
    lens = torch.from_numpy(w["seq_lens"]).to(dev)
    if sparse:
        # The plan depends on B, H and topk only; lists and lengths are read
        # on the device. A step: gather kernel, decode kernel (+ combine).
        topk_dev = torch.from_numpy(w["topk_indices"]).to(dev)
        plan = m.mla_sparse_plan(B, H, int(w["topk_indices"].shape[1]))
        launches_per_step = 2 + (1 if any(plan.num_splits(b) > 1 for b in range(B)) else 0)
    else:
        plan = m.mla_decode_plan(B, heads, w["seq_lens"], bs, int(w["max_blocks"]), q_len=q_len,
                                 lengths_are_bounds=args.graph)
    out = torch.empty(plan.q_shape(512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty(plan.q_shape(None), dtype=torch.float32, device=dev)
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=dev)
    if not sparse:
        launches_per_step = 1 + (1 if plan.workspace_bytes else 0)
    stream = torch.cuda.current_stream()

    def call(st):
        if sparse:
            m.mla_decode_sparse(plan, q_nope, q_pe, kv, table, lens, topk_dev, w["sm_scale"], out,
                                lse, ws, kv_scale=w["kv_scale"] if fp8 else None, stream=st)
        elif fp8:
            m.mla_decode_fp8(plan, q_nope, q_pe, kv, w["kv_scale"], table, lens, w["sm_scale"], out,
                             lse, ws, st)
        else:
            m.mla_decode(plan, q_nope, q_pe, kv, table, lens, w["sm_scale"], out, lse, ws, st)

    def step():
        call(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert m.mla_check_device_error(plan) == 0
    if args.graph:
        # One step captured on a side stream; every timed step replays it on
        # the launching stream.
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            call(cap)
        cap.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            call(cap)
        torch.cuda.synchronize()

        def step():  # noqa: F811 (the timed step is the replay)
            graph.replay()

        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        assert m.mla_check_device_error(plan) == 0

    # A cache several times the L2 size leaves no reuse between steps; a
    # smaller one gets L2 flushed (a write larger than L2) before every step,
    # outside the timed events of that step.
    cache_bytes = int(cache_of(w).nbytes)
    flush = None
    if cache_bytes < 4 * L2_BYTES:
        flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(dist)
    torch.cuda.synchronize()
    for i in range(args.steps):
        if flush is not None:
            flush.fill_(i & 0xFF)
        ev0[i].record(stream)
        step()
        ev1[i].record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    clocks = sampler.stop()
    per_step = [ev0[i].elapsed_time(ev1[i]) for i in range(args.steps)]
    total_ms = sum(per_step)
    total_ms = max_over_ranks(total_ms, dist, dev)
    ms_per_step = total_ms / args.steps
    us = ms_per_step * 1e3
    assert m.mla_check_device_error(plan) == 0

    # End to end through the public API with host buffers: pinned host inputs
    # of the step (queries, block table, lengths) copied in, plan rebuilt from
    # the host lengths, decode, and out + lse copied back. The cache is state
    # resident on the device across steps, as in serving.
    h_qn = torch.from_numpy(w["q_nope"].view(np.int16)).view(torch.bfloat16).pin_memory()
    h_qp = torch.from_numpy(w["q_pe"].view(np.int16)).view(torch.bfloat16).pin_memory()
    h_tab = torch.from_numpy(w["block_table"]).pin_memory()
    h_len = torch.from_numpy(w["seq_lens"]).pin_memory()
    h_idx = torch.from_numpy(w["topk_indices"]).pin_memory() if sparse else None
    h_out = torch.empty(tuple(out.shape), dtype=torch.bfloat16).pin_memory()
    h_lse = torch.empty(tuple(lse.shape), dtype=torch.float32).pin_memory()
    lens_np = w["seq_lens"].copy()
    e_steps = max(3, min(args.steps, 20))

    def copies_in():
        q_nope.copy_(h_qn, non_blocking=True)
        q_pe.copy_(h_qp, non_blocking=True)
        table.copy_(h_tab, non_blocking=True)
        lens.copy_(h_len, non_blocking=True)
        if sparse:
            topk_dev.copy_(h_idx, non_blocking=True)

    def e2e_step():
        copies_in()
        if not sparse and not args.graph:   # sparse and bounds plans serve any lengths
            plan.update(lens_np, stream)
        step()
        h_out.copy_(out, non_blocking=True)
        h_lse.copy_(lse, non_blocking=True)
        stream.synchronize()

    for _ in range(2):
        e2e_step()
    barrier(dist)
    t_e = time.perf_counter()
    for _ in range(e_steps):
        e2e_step()
    e2e_ms = (time.perf_counter() - t_e) * 1e3 / e_steps
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)

    # Where an end-to-end step goes, from separate passes outside the timed
    # loop: device time of the input copies, the decode and the output copies
    # (CUDA events on the stream, each phase alone), and the host time of the
    # plan update (which overlaps the input copies in the step above).
    def phase_us(fn, n=5):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]
        for a, b in ev:
            a.record(stream)
            fn()
            b.record(stream)
            stream.synchronize()
        return statistics.median(a.elapsed_time(b) * 1e3 for a, b in ev)


    def copies_out():
        h_out.copy_(out, non_blocking=True)
        h_lse.copy_(lse, non_blocking=True)

    plan_host_us = 0.0
    if not sparse and not args.graph:
        t_p = time.perf_counter()
        for _ in range(5):
            plan.update(lens_np, stream)
        stream.synchronize()
        plan_host_us = (time.perf_counter() - t_p) * 1e6 / 5
    breakdown = {"h2d_us": round(phase_us(copies_in), 1),
                 "plan_update_host_us": round(plan_host_us, 1),
                 "decode_us": round(phase_us(step), 1),
                 "d2h_us": round(phase_us(copies_out), 1)}
    h2d = sum(t.numel() * t.element_size()
              for t in (h_qn, h_qp, h_tab, h_len) + ((h_idx,) if sparse else ()))
    d2h = h_out.numel() * h_out.element_size() + h_lse.numel() * h_lse.element_size()

    peaks, peak_kind = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    tf = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    t_bytes_us = counts["bytes"] / (hbm * 1e9) * 1e6
    # FLOPs at the dense bf16 peak (the roofline_fraction below); the bound
    # itself takes the contraction's own dtype: e4m3 for an FP8 cache.
    t_flops_bf16_us = counts["flops"] / (tf * 1e12) * 1e6
    tf_own = tf * (FP8_OVER_BF16 if fp8 else 1.0)
    t_flops_us = counts["flops"] / (tf_own * 1e12) * 1e6
    # Dominant kernel: the decode kernel. Without a split the step is exactly
    # that one launch, so the step time is its duration. A sparse step also
    # runs the gather kernel; its bound is taken over the whole step.
    dominant_us = us if launches_per_step == 1 else None
    hbm_bound = t_bytes_us >= t_flops_us
    achieved = (counts["bytes"] / (ms_per_step * 1e-3) / 1e9 if hbm_bound
                else counts["flops"] / (ms_per_step * 1e-3) / 1e12)
    traffic = recorded_traffic(args.config, args.kv)
    result = {
        "metric": METRIC,
        "value": round(us, 2),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3" if fp8 else "bf16",
        "data": ("synthetic (seeded N(0,1) latent cache quantised to E4M3 with scale "
                 f"{w['kv_scale']}, bf16 queries, sentinel-filled spare blocks and tail slots)"
                 if fp8 else
                 "synthetic (seeded N(0,1) bf16 latent cache and queries, sentinel-filled spare "
                 "blocks and tail slots)"),
        "config": workload_config(spec, w, counts, world, args.graph),
        "plan": {"cta_pairs": plan.num_clusters, "work_items": plan.num_work_items,
                 "split_requests": int(sum(plan.num_splits(b) > 1 for b in range(B)))},
        "kv_read_gbs": round(counts["kv_bytes"] / (ms_per_step * 1e-3) / 1e9, 1),
        "alg_bytes_per_call": counts["bytes"],
        "alg_flops_per_call": counts["flops"],
        "roofline": {
            "bound": "hbm" if hbm_bound else "tensor",
            "achieved": round(achieved, 1),
            "peak": hbm if hbm_bound else tf_own,
            "unit": "GB/s" if hbm_bound else "TFLOP/s",
            "frac": round(achieved / (hbm if hbm_bound else tf_own), 4),
            "peak_source": (f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if hbm_bound else
                            f"{peak_kind} (MEASURED_PEAKS.json bf16_tflops"
                            + (" x 2, the nominal fp8/bf16 ratio)" if fp8 else ")"))
                           if peak_kind == "measured" else "fallback 6.8 TB/s, 1.9 PFLOP/s",
            "traffic": traffic,
            "t_bytes_us": round(t_bytes_us, 2),
            "t_flops_us": round(t_flops_us, 2),
            "t_flops_bf16_us": round(t_flops_bf16_us, 2),
            "roofline_fraction": round(max(t_bytes_us, t_flops_bf16_us) / us, 4),
            "dominant_kernel": "mla_decode_kernel",
            "scope": ("whole step: sparse gather + decode" + (" + combine" if launches_per_step > 2
                                                               else "")) if sparse else
                     ("decode kernel" if launches_per_step == 1 else "decode + combine"),
            "dominant_kernel_us": round(dominant_us, 2) if dominant_us else None,
        },
        "step_us_min": round(min(per_step) * 1e3, 2),
        "step_us_median": round(statistics.median(per_step) * 1e3, 2),
        "e2e": {"value": round(e2e_ms * 1e3, 2), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "breakdown": breakdown},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu:
        result["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    if dist is not None:
        dist.destroy_process_group()
    return result if rank == 0 else None


# ------------------------------------------------------------- CPU oracle leg

def oracle_call(oracle, w, reqs=None):
    """The oracle on requests `reqs` (all when None) of workload w."""
    sel = slice(None) if reqs is None else np.asarray(reqs)
    qn, qp = w["q_nope"][sel], w["q_pe"][sel]
    bt, sl = w["block_table"][sel], w["seq_lens"][sel]
    if "q_len" in w and "kv_fp8" not in w:
        return oracle.mla_decode_multi(qn, qp, w["kv_cache"], bt, sl, w["sm_scale"])
    if "topk_indices" in w:
        idx = w["topk_indices"][sel]
        if "kv_fp8" in w:
            return oracle.mla_decode_sparse(qn, qp, None, bt, sl, idx, w["sm_scale"],
                                            kv_fp8=w["kv_fp8"], kv_scale=w["kv_scale"])
        return oracle.mla_decode_sparse(qn, qp, w["kv_cache"], bt, sl, idx, w["sm_scale"])
    if "kv_fp8" in w:
        return oracle.mla_decode_fp8(qn, qp, w["kv_fp8"], w["kv_scale"], bt, sl, w["sm_scale"])
    return oracle.mla_decode(qn, qp, w["kv_cache"], bt, sl, w["sm_scale"])


def sample_requests(rng, seq, n):
    """n random requests with at least one token (all of them if fewer)."""
    nz = np.nonzero(seq > 0)[0]
    return np.sort(rng.permutation(nz)[:max(1, min(n, nz.size))])


def cpu_baseline(w, budget_s: float):
    """The fp64 oracle as it stands, on a bounded random sample of the
    workload's requests (all their heads), scaled to one full call by the
    sample's share of the tokens."""
    import oracle
    oracle.build()
    B, H = int(w["B"]), int(w["H"])
    cores = oracle.num_threads(0)
    seq = request_work(w)
    rng = np.random.default_rng(123)
    reqs = sample_requests(rng, seq, max(1, cores // max(1, H // 16)))
    t0 = time.perf_counter()
    oracle_call(oracle, w, reqs)
    pilot = time.perf_counter() - t0
    n2 = int(min(B, max(reqs.size, reqs.size * budget_s / max(pilot, 1e-6))))
    reqs = sample_requests(rng, seq, n2)
    t0 = time.perf_counter()
    oracle_call(oracle, w, reqs)
    dt = time.perf_counter() - t0
    share = seq[reqs].sum() / seq.sum()
    per_call_s = dt / share
    return {"value": round(per_call_s * 1e6, 1), "unit": UNIT, "cores": int(cores), "kind": "oracle",
            "sample": f"{reqs.size} of {B} requests (all {H} query rows each), {dt:.1f} s, scaled by "
                      f"token share {share:.4f}"}


def bench_reference(args, world, rank, local):
    """--impl reference: the oracle on the host cores, each step the whole
    workload when the run fits the time budget, else a bounded sample."""
    if world > 1:
        init_dist(world, "gloo")
        if rank != 0:
            return None
    spec = spec_of(args.config)
    w = load_workload(args.config, args.kv, args.q_len)
    import oracle
    oracle.build()
    B, H = int(w["B"]), int(w["H"])
    cores = oracle.num_threads(0)
    seq = request_work(w)
    rng = np.random.default_rng(7)
    total_steps = args.warmup + args.steps
    # Pilot: a few requests, to size the steps; when that puts one whole call
    # under 20 s, one whole call times it directly (a small sample runs below
    # the oracle's full parallel rate and overestimates it).
    pilot = sample_requests(rng, seq, max(1, cores // max(1, H // 16)))
    t0 = time.perf_counter()
    oracle_call(oracle, w, pilot)
    pilot_s = time.perf_counter() - t0
    full_est_s = pilot_s / max(seq[pilot].sum() / max(seq.sum(), 1), 1e-12)
    if full_est_s < 20.0:
        t0 = time.perf_counter()
        oracle_call(oracle, w)
        full_est_s = time.perf_counter() - t0
    budget_s = 300.0
    full = total_steps * full_est_s <= budget_s
    times = []
    if full:
        # Every step is one whole call of the oracle on the workload.
        for s in range(total_steps):
            t0 = time.perf_counter()
            oracle_call(oracle, w)
            dt = time.perf_counter() - t0
            if s >= args.warmup:
                times.append(dt)
        sample = f"the full workload every step ({B} requests x {H} query rows)"
    else:
        # Each step: a random sample of requests sized so the run stays within
        # the budget, scaled by its token share to one call.
        n_req = int(max(1, min(B, (budget_s / max(total_steps, 1)) / max(full_est_s, 1e-9) * B)))
        for s in range(total_steps):
            reqs = sample_requests(rng, seq, n_req)
            t0 = time.perf_counter()
            oracle_call(oracle, w, reqs)
            dt = time.perf_counter() - t0
            if s >= args.warmup:
                times.append(dt / (seq[reqs].sum() / seq.sum()))
        sample = (f"{n_req} random requests (all {H} query rows) per step, scaled by token share to "
                  "one full call (the full call would not fit the run's time budget)")
    us = statistics.mean(times) * 1e6
    return {
        "impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(us / 1e3, 3), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(spec, w, counts_of(w), world, args.graph),
        "cpu_baseline": {"value": round(us, 1), "unit": UNIT, "cores": int(cores), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(us, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=DEFAULT_CONFIG,
                    choices=sorted(list(wl.WORKLOADS_BY_NAME) + list(wl.SPARSE_WORKLOADS)))
    ap.add_argument("--kv", choices=["bf16", "fp8"], default="bf16",
                    help="cache element type (fp8: E4M3 with a per-tensor scale)")
    ap.add_argument("--q-len", type=int, default=1,
                    help="query tokens per request (speculative decoding; dense workloads)")
    ap.add_argument("--graph", action="store_true",
                    help="time CUDA-graph replays of one captured step (length-bounds plan)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline leg")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_env()
    if world != args.gpus and world > 1:
        log(f"[bench] WORLD_SIZE={world} differs from --gpus {args.gpus}; using WORLD_SIZE")
    fn = bench_reference if args.impl == "reference" else bench_ours
    res = fn(args, world, rank, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
