"""Seeded synthetic inputs for paged MLA decode.

This module is the one piece both sides of the parity tests share: it builds
the host arrays that the CUDA library and the CPU oracle both receive. It holds
no arithmetic of the method itself (no scores, softmax or reductions), only
random draws, bf16 rounding of those draws, and the placement of blocks in the
paged cache.

Shapes follow the pages' decode setting: a paged latent cache of 576-wide bf16
rows (512 c_kv followed by 64 k_pe) addressed through an int32 block table, as
served with ``--block-size 32`` in "[Kernel] Flashinfer MLA (trtllm-gen) decode
kernel integration" (vLLM PR #21078), E2E Benchmark, with DeepSeek-R1 head
count 128 and the fewer-than-128-head case of "SM100 Cutlass MLA decode with
unrestricted num_heads (< 128) for DeepSeek TP" (vLLM PR #20769).

Recipe (every draw comes from one ``numpy.random.PCG64(seed)`` stream in a
fixed order):
  1. sequence lengths from the workload's rule (inclusive integer ranges);
  2. a random permutation of the physical block pool; each request's pages
     take the next blocks of the permutation in order, the rest are spare;
  3. every cached element of a used block ~ N(0, 1), rounded to bf16 (RNE);
  4. q_nope, q_pe ~ N(0, 1) rounded to bf16;
  5. sentinels: every element of a spare block and of the unused tail slots of
     each request's last page is bf16(+-1e4) = +-9984 with a random sign, so a
     kernel that reads past a sequence's end or an unused block is caught;
  6. block-table entries past a request's last page point at random spare
     blocks (never -1, so a faulty reader sees sentinels instead of faulting);
  7. optionally ("peaky" rows) each valid token row is multiplied by 8 with
     probability 0.01 (exact in bf16).

FP8 variant (``to_fp8``): the same workload with its cache stored as OCP E4M3
bytes under one per-tensor scale, as an engine serving with an fp8 KV cache
would hold it: byte = E4M3 round-to-nearest-even of (element / kv_scale),
clipped to the largest finite magnitude 448, so the sentinels become +-448
(standing for +-448 * kv_scale) and the N(0, 1) rows keep 4 significant bits.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Callable, Dict, List, Optional, Sequence

import numpy as np

D_C = 512
D_R = 64
D = D_C + D_R
SENTINEL_BF16 = 0x461C       # bf16 bits of 9984.0 = bf16(1e4); 0xC61C is -9984.0
SM_SCALE_192 = 1.0 / math.sqrt(192.0)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest even); returns uint16 bits.

    Inputs here are finite random draws, so no NaN handling is needed.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass(frozen=True)
class WorkloadSpec:
    name: str
    B: int
    H: int
    block_size: int
    seed: int
    seq_lens: Callable[[np.random.Generator], np.ndarray]
    max_len: int                      # upper bound of the length rule -> max_blocks
    pool: Callable[[int], int]        # required blocks -> pool size
    peaky_fraction: float = 0.0       # fraction of valid rows scaled by 8
    sm_scale: float = SM_SCALE_192
    description: str = ""


def _pool_125(required: int) -> int:
    return max(int(math.ceil(1.25 * required)), required + 4)


def _fixed_lens(values: Sequence[int]):
    arr = np.asarray(values, dtype=np.int32)
    return lambda rng: arr.copy()


def _uniform_lens(B: int, lo: int, hi: int):
    return lambda rng: rng.integers(lo, hi, size=B, endpoint=True).astype(np.int32)


# The five decode configurations. Index 0 is the small case the oracle finishes
# in seconds; index 3 is the B=512, H=128 high-concurrency shape.
WORKLOADS: List[WorkloadSpec] = [
    WorkloadSpec("tiny_b2_h16", B=2, H=16, block_size=32, seed=1,
                 seq_lens=_fixed_lens([1, 256]), max_len=256,
                 pool=lambda req: req + 4,
                 description="B=2, H=16, L=[1,256], bs=32, 4 spare sentinel blocks"),
    WorkloadSpec("v2lite_b64_h16", B=64, H=16, block_size=64, seed=2,
                 seq_lens=_uniform_lens(64, 1, 4096), max_len=4096, pool=_pool_125,
                 description="B=64, H=16, L~U{1..4096}, bs=64, pool 1.25x required"),
    WorkloadSpec("r1_b128_h128", B=128, H=128, block_size=32, seed=3,
                 seq_lens=_uniform_lens(128, 1024, 3072), max_len=3072, pool=_pool_125,
                 description="B=128, H=128, L=1024+U{0..2048}, bs=32, pool 1.25x required"),
    WorkloadSpec("r1_b512_h128", B=512, H=128, block_size=32, seed=4,
                 seq_lens=_uniform_lens(512, 1024, 3072), max_len=3072,
                 pool=lambda req: max(35265, req + 4),
                 description="B=512, H=128, L=1024+U{0..2048}, bs=32, 35265-block (~1.3 GB) pool"),
    WorkloadSpec("long_b4_h128", B=4, H=128, block_size=64, seed=5,
                 seq_lens=_fixed_lens([65536, 32768, 8191, 1]), max_len=65536,
                 pool=_pool_125, peaky_fraction=0.01,
                 description="B=4, H=128, L=[65536,32768,8191,1], bs=64, 1% rows x8"),
]
WORKLOADS_BY_NAME: Dict[str, WorkloadSpec] = {w.name: w for w in WORKLOADS}

# Sparse (top-k) decode: a long-context R1-shaped batch in which every request
# attends to 2048 of its tokens (the token selection itself happens upstream).
SPARSE_TOPK = 2048
SPARSE_WORKLOADS: Dict[str, WorkloadSpec] = {
    "sparse_r1_b64_h128": WorkloadSpec(
        "sparse_r1_b64_h128", B=64, H=128, block_size=64, seed=6,
        seq_lens=_uniform_lens(64, 8192, 16384), max_len=16384, pool=_pool_125,
        description="B=64, H=128, L=8192+U{0..8192}, bs=64, top-2048 selection per request"),
    # The same recipe at a quarter of the requests: the case profiled with
    # multi-pass counters (a 230 MB cache, above the L2 size).
    "sparse_r1_b16_h128": WorkloadSpec(
        "sparse_r1_b16_h128", B=16, H=128, block_size=64, seed=7,
        seq_lens=_uniform_lens(16, 8192, 16384), max_len=16384, pool=_pool_125,
        description="B=16, H=128, L=8192+U{0..8192}, bs=64, top-2048 selection per request"),
}


def multi_token(spec: WorkloadSpec, q_len: int) -> Dict[str, object]:
    """The workload of ``spec`` with q_len query tokens per request (the
    speculative-decoding shape): the generator's draws for q_len * H query
    rows, viewed as [B, q_len, H, ...] (``q_len`` and ``heads`` keys added).
    The lengths count the q_len new tokens, so every L must be >= q_len."""
    w = dict(generate(dataclasses.replace(spec, H=spec.H * q_len, name=f"{spec.name}_q{q_len}")))
    w["q_len"], w["heads"] = int(q_len), int(spec.H)
    w["q_nope"] = w["q_nope"].reshape(spec.B, q_len, spec.H, D_C)
    w["q_pe"] = w["q_pe"].reshape(spec.B, q_len, spec.H, D_R)
    return w


def custom_spec(name: str, B: int, H: int, block_size: int, seq_lens: Sequence[int],
                seed: int, spare_blocks: int = 4, peaky_fraction: float = 0.0,
                max_blocks: Optional[int] = None,
                sm_scale: float = SM_SCALE_192) -> WorkloadSpec:
    """A small workload with explicit lengths (edge cases in the tests)."""
    lens = list(seq_lens)
    max_len = max(lens) if lens else 0
    if max_blocks is not None:
        max_len = max(max_len, max_blocks * block_size)
    return WorkloadSpec(name, B=B, H=H, block_size=block_size, seed=seed,
                        seq_lens=_fixed_lens(lens), max_len=max_len,
                        pool=lambda req: req + spare_blocks, peaky_fraction=peaky_fraction,
                        sm_scale=sm_scale)


def _normal_bf16(rng: np.random.Generator, n: int, chunk: int = 1 << 24) -> np.ndarray:
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = f32_to_bf16_bits(rng.standard_normal(e - s, dtype=np.float32))
    return out


def generate(spec: WorkloadSpec) -> Dict[str, object]:
    """Build the seeded host arrays of one workload (see the module recipe)."""
    rng = np.random.Generator(np.random.PCG64(spec.seed))
    bs = spec.block_size
    seq_lens = np.asarray(spec.seq_lens(rng), dtype=np.int32)
    assert seq_lens.shape == (spec.B,)
    pages = (seq_lens.astype(np.int64) + bs - 1) // bs
    required = int(pages.sum())
    max_blocks = max(1, int(math.ceil(spec.max_len / bs)))
    assert int(pages.max(initial=0)) <= max_blocks
    num_blocks = int(spec.pool(required))
    assert num_blocks > required, "need at least one spare (sentinel) block"

    perm = rng.permutation(num_blocks).astype(np.int32)
    used, spare = perm[:required], perm[required:]

    kv = _normal_bf16(rng, num_blocks * bs * D).reshape(num_blocks, bs, D)
    q_nope = _normal_bf16(rng, spec.B * spec.H * D_C).reshape(spec.B, spec.H, D_C)
    q_pe = _normal_bf16(rng, spec.B * spec.H * D_R).reshape(spec.B, spec.H, D_R)

    block_table = np.empty((spec.B, max_blocks), dtype=np.int32)
    cursor = 0
    for b in range(spec.B):
        n = int(pages[b])
        block_table[b, :n] = used[cursor:cursor + n]
        cursor += n
        if n < max_blocks:
            block_table[b, n:] = spare[rng.integers(0, spare.shape[0], size=max_blocks - n)]

    # Sentinels: spare blocks entirely, then each request's unused tail slots.
    sign = rng.integers(0, 2, size=(spare.shape[0], bs, D), dtype=np.uint16)
    kv[spare] = np.uint16(SENTINEL_BF16) | (sign << np.uint16(15))
    for b in range(spec.B):
        L = int(seq_lens[b])
        if L == 0 or L % bs == 0:
            continue
        blk = block_table[b, L // bs]
        tail = bs - L % bs
        s = rng.integers(0, 2, size=(tail, D), dtype=np.uint16)
        kv[blk, L % bs:] = np.uint16(SENTINEL_BF16) | (s << np.uint16(15))

    if spec.peaky_fraction > 0.0:
        for b in range(spec.B):
            L = int(seq_lens[b])
            hit = np.nonzero(rng.random(L) < spec.peaky_fraction)[0]
            for t in hit:
                blk, slot = block_table[b, t // bs], t % bs
                row = bf16_bits_to_f32(kv[blk, slot]) * np.float32(8.0)
                kv[blk, slot] = f32_to_bf16_bits(row)   # exact: a power-of-two scale

    return {
        "name": spec.name,
        "B": spec.B,
        "H": spec.H,
        "block_size": bs,
        "num_blocks": num_blocks,
        "max_blocks": max_blocks,
        "seq_lens": seq_lens,
        "block_table": block_table,
        "kv_cache": kv,
        "q_nope": q_nope,
        "q_pe": q_pe,
        "sm_scale": float(spec.sm_scale),
        "spare_blocks": np.sort(spare),
    }


FP8_KV_SCALE = 0.1            # per-tensor scale of the FP8 workloads (not a power of two)
E4M3_MAX = 448.0


def to_fp8(w: Dict[str, object], kv_scale: float = FP8_KV_SCALE) -> Dict[str, object]:
    """The workload with its cache quantised to E4M3 bytes (see the recipe).

    Adds ``kv_fp8`` (uint8, same shape as ``kv_cache``) and ``kv_scale``; the
    bf16 ``kv_cache`` is dropped. Rounding uses torch's float8_e4m3fn cast
    (round to nearest even) after clipping to +-448.
    """
    import torch
    src = w["kv_cache"].reshape(-1)
    codes = np.empty(src.shape, dtype=np.uint8)
    step = 1 << 24
    for s in range(0, src.size, step):   # in chunks: the full cache is ~650M elements
        x = bf16_bits_to_f32(src[s:s + step]) / np.float32(kv_scale)
        np.clip(x, -E4M3_MAX, E4M3_MAX, out=x)
        codes[s:s + step] = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    out = {k: v for k, v in w.items() if k != "kv_cache"}
    out["kv_fp8"] = codes.reshape(w["kv_cache"].shape)
    out["kv_scale"] = float(kv_scale)
    out["name"] = f"{w['name']}_fp8"
    return out


def with_topk(w: Dict[str, object], topk: int, seed: int,
              mixed_padding: bool = False) -> Dict[str, object]:
    """Adds ``topk_indices`` (int32 [B, topk]) to a workload: for each request,
    min(topk, L) distinct token positions drawn uniformly without replacement,
    in random order, the remaining entries padding (-1 at the end). With
    ``mixed_padding`` the padding entries are -1 or L + k (k < 7) at random and
    the whole row is shuffled, so padding sits between selected tokens. Draws
    come from ``numpy.random.PCG64(seed)``."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lens = np.asarray(w["seq_lens"], dtype=np.int64)
    B = lens.shape[0]
    idx = np.full((B, topk), -1, dtype=np.int32)
    for b in range(B):
        L = int(lens[b])
        n = min(topk, L)
        row = np.full(topk, -1, dtype=np.int64)
        if n > 0:
            row[:n] = rng.choice(L, size=n, replace=False)
        if mixed_padding:
            if n < topk:
                pads = rng.integers(0, 2, size=topk - n)
                row[n:] = np.where(pads == 0, -1, L + rng.integers(0, 7, size=topk - n))
            row = row[rng.permutation(topk)]
        idx[b] = row.astype(np.int32)
    out = dict(w)
    out["topk_indices"] = idx
    out["topk"] = topk
    return out


def permute_blocks(w: Dict[str, object], seed: int) -> Dict[str, object]:
    """Same logical cache under a different physical block placement.

    Physical block i moves to slot pi[i]; every table entry is remapped, so
    request b still sees the same rows in the same order.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    nb = int(w["num_blocks"])
    pi = rng.permutation(nb).astype(np.int32)
    key = "kv_fp8" if "kv_fp8" in w else "kv_cache"
    kv = np.empty_like(w[key])
    kv[pi] = w[key]
    out = dict(w)
    out[key] = kv
    out["block_table"] = pi[w["block_table"]]
    out["spare_blocks"] = np.sort(pi[w["spare_blocks"]])
    return out


def expected_counts(w: Dict[str, object]) -> Dict[str, float]:
    """Algorithmic byte and flop counts of one decode call on this workload.

    Bytes: KV rows read once (1152 B each, 576 B for an FP8 cache), q_nope+q_pe, out (bf16), lse (fp32),
    the block-table entries of used pages and the lengths. Flops: per token and
    real head, 2*576 for the score and 2*512 for the value product.
    """
    seq = np.asarray(w["seq_lens"], dtype=np.int64)
    B, H, bs = int(w["B"]), int(w["H"]), int(w["block_size"])
    tokens = int(seq.sum())
    pages = int(((seq + bs - 1) // bs).sum())
    kv_bytes = tokens * D * (1 if "kv_fp8" in w else 2)
    total = kv_bytes + B * H * D * 2 + B * H * D_C * 2 + 4 * B * H + 4 * pages + 4 * B
    q_len = int(w.get("q_len", 1))
    if q_len == 1:
        flops = tokens * H * (2 * D + 2 * D_C)
    else:   # H = q_len * heads rows; query token j sees the first L - q_len + 1 + j tokens
        heads = H // q_len
        seen = sum(max(0, int(L) - q_len + 1 + j) for L in seq for j in range(q_len))
        flops = seen * heads * (2 * D + 2 * D_C)
    return {"tokens": tokens, "kv_bytes": float(kv_bytes), "bytes": float(total),
            "flops": float(flops)}


def sparse_counts(w: Dict[str, object]) -> Dict[str, float]:
    """Algorithmic byte and flop counts of one sparse decode call: the cache
    rows of the valid list entries read once (a duplicate counts each time),
    the block-table entry of each, the lists themselves, q_nope+q_pe, out,
    lse and the lengths. Flops as for the dense decode, over the valid
    entries."""
    seq = np.asarray(w["seq_lens"], dtype=np.int64)
    idx = np.asarray(w["topk_indices"], dtype=np.int64)
    B, H = int(w["B"]), int(w["H"])
    tokens = int(((idx >= 0) & (idx < seq[:, None])).sum())
    kv_bytes = tokens * D * (1 if "kv_fp8" in w else 2)
    total = (kv_bytes + 4 * tokens + 4 * idx.size + B * H * D * 2 + B * H * D_C * 2 + 4 * B * H
             + 4 * B)
    flops = tokens * H * (2 * D + 2 * D_C)
    return {"tokens": tokens, "kv_bytes": float(kv_bytes), "bytes": float(total),
            "flops": float(flops)}
