"""fp64 CPU oracle for paged MLA decode (ctypes wrapper over ``mla_oracle.cpp``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` are the only code allowed to import this package.
It never imports the CUDA library package and the CUDA library never imports
it.

Inputs are the same host arrays the GPU path receives: bf16 tensors as
``numpy.uint16`` bit patterns, int32 block tables and sequence lengths.
Outputs are float64.

Where the definition comes from: "SM100 Cutlass MLA decode with unrestricted
num_heads (< 128) for DeepSeek TP" (vLLM PR #20769), bot summary (split KV
plus a reduction kernel) and "[Kernel] Flashinfer MLA (trtllm-gen) decode
kernel integration" (vLLM PR #21078), E2E Benchmark (paged cache,
--block-size 32). The C++ file's header states the computation step by step.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.cpp")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_mla.so")

D_C = 512
D_R = 64
D = D_C + D_R

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library with g++ (OpenMP, -O2) if needed."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-std=c++17", "-O2", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        p = ctypes.c_void_p
        i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        common = [i32, i32, p, p, p, i64, i32, p, i32, p, dbl]
        lib.oracle_mla_decode_rows.argtypes = common + [i64, p, p, p, p, i32]
        lib.oracle_mla_decode.argtypes = common + [p, p, i32]
        lib.oracle_mla_decode_multi.argtypes = [i32, i32, i32, p, p, p, i64, i32, p, i32, p, dbl,
                                                p, p, i32]
        lib.oracle_mla_partial.argtypes = common + [i32, i32, i64, i64, p, p]
        lib.oracle_mla_combine.argtypes = [i32, p, p, p, p]
        lib.oracle_mla_decode_bruteforce.argtypes = common + [p, p]
        lib.oracle_mla_decode_fp8.argtypes = [i32, i32, i32, p, p, p, dbl, i64, i32, p, i32, p,
                                              dbl, p, p, i32]
        lib.oracle_e4m3_decode.argtypes = [i64, p, p]
        lib.oracle_mla_decode_sparse.argtypes = [i32, i32, p, p, p, i64, i32, p, i32, p, p, i32,
                                                 dbl, p, p, i32, p, dbl]
        lib.oracle_mla_decode_sparse.restype = ctypes.c_int
        lib.oracle_num_threads.argtypes = [i32]
        for fn in (lib.oracle_mla_decode_rows, lib.oracle_mla_decode, lib.oracle_mla_decode_multi,
                   lib.oracle_mla_decode_fp8, lib.oracle_e4m3_decode,
                   lib.oracle_mla_partial,
                   lib.oracle_mla_combine, lib.oracle_mla_decode_bruteforce,
                   lib.oracle_num_threads):
            fn.restype = ctypes.c_int
        _lib = lib
        return lib


class OracleError(RuntimeError):
    pass


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise OracleError(f"{what} failed with code {rc} "
                          "(1 = bad argument, 2 = block id out of range)")


def _common(q_nope, q_pe, kv_cache, block_table, seq_lens, sm_scale):
    q_nope = np.ascontiguousarray(q_nope, dtype=np.uint16)
    q_pe = np.ascontiguousarray(q_pe, dtype=np.uint16)
    kv_cache = np.ascontiguousarray(kv_cache, dtype=np.uint16)
    block_table = np.ascontiguousarray(block_table, dtype=np.int32)
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, H, dc = q_nope.shape
    assert dc == D_C and q_pe.shape == (B, H, D_R), (q_nope.shape, q_pe.shape)
    nb, bs, d = kv_cache.shape
    assert d == D, kv_cache.shape
    assert block_table.ndim == 2 and block_table.shape[0] == B
    assert seq_lens.shape == (B,)
    args = (B, H, _ptr(q_nope), _ptr(q_pe), _ptr(kv_cache), nb, bs, _ptr(block_table),
            block_table.shape[1], _ptr(seq_lens), float(sm_scale))
    keep = (q_nope, q_pe, kv_cache, block_table, seq_lens)
    return args, keep


def num_threads(n_threads: int = 0) -> int:
    """OpenMP thread count the oracle uses (n_threads <= 0: runtime default)."""
    return _load().oracle_num_threads(int(n_threads))


def mla_decode(q_nope, q_pe, kv_cache, block_table, seq_lens, sm_scale, n_threads: int = 0):
    """Full decode: returns (out[B, H, 512] float64, lse[B, H] float64)."""
    args, keep = _common(q_nope, q_pe, kv_cache, block_table, seq_lens, sm_scale)
    B, H = args[0], args[1]
    out = np.empty((B, H, D_C), dtype=np.float64)
    lse = np.empty((B, H), dtype=np.float64)
    _check(_load().oracle_mla_decode(*args, _ptr(out), _ptr(lse), int(n_threads)),
           "oracle_mla_decode")
    del keep
    return out, lse


def mla_decode_multi(q_nope, q_pe, kv_cache, block_table, seq_lens, sm_scale, n_threads: int = 0):
    """Multi-token (speculative) decode: q_nope [B, q_len, H, 512], q_pe
    [B, q_len, H, 64]; query token j of request b attends to its first
    L - q_len + 1 + j tokens. Returns (out [B, q_len, H, 512], lse [B, q_len, H])."""
    q_nope = np.ascontiguousarray(q_nope, dtype=np.uint16)
    q_pe = np.ascontiguousarray(q_pe, dtype=np.uint16)
    B, q_len, H, dc = q_nope.shape
    assert dc == D_C and q_pe.shape == (B, q_len, H, D_R), (q_nope.shape, q_pe.shape)
    args, keep = _common(q_nope.reshape(B, q_len * H, D_C), q_pe.reshape(B, q_len * H, D_R),
                         kv_cache, block_table, seq_lens, sm_scale)
    out = np.empty((B, q_len, H, D_C), dtype=np.float64)
    lse = np.empty((B, q_len, H), dtype=np.float64)
    (_, _, qn, qp, kv, nb, bs, bt, mb, sl, sc) = args
    _check(_load().oracle_mla_decode_multi(B, q_len, H, qn, qp, kv, nb, bs, bt, mb, sl, sc,
                                           _ptr(out), _ptr(lse), int(n_threads)),
           "oracle_mla_decode_multi")
    del keep
    return out, lse


def mla_decode_sparse(q_nope, q_pe, kv_cache, block_table, seq_lens, topk_indices, sm_scale,
                      n_threads: int = 0, kv_fp8=None, kv_scale: float = 1.0):
    """Sparse decode: request b attends to the tokens topk_indices[b] (int32
    [B, topk]; entries outside [0, L) are padding). With ``kv_fp8`` (uint8 E4M3
    bytes, same shape as a cache) the cache is that FP8 one with ``kv_scale``
    and ``kv_cache`` may be None. Returns (out, lse) float64."""
    f8 = None
    if kv_fp8 is not None:
        f8 = np.ascontiguousarray(kv_fp8, dtype=np.uint8)
        kv_cache = np.zeros((1, f8.shape[1], D), dtype=np.uint16)   # shape check only
    args, keep = _common(q_nope, q_pe, kv_cache, block_table, seq_lens, sm_scale)
    B, H = args[0], args[1]
    if f8 is not None:
        args = args[:5] + (f8.shape[0],) + args[6:]
    idx = np.ascontiguousarray(topk_indices, dtype=np.int32)
    assert idx.ndim == 2 and idx.shape[0] == B, idx.shape
    out = np.empty((B, H, D_C), dtype=np.float64)
    lse = np.empty((B, H), dtype=np.float64)
    (_, _, qn, qp, kv, nb, bs, bt, mb, sl, sc) = args
    _check(_load().oracle_mla_decode_sparse(B, H, qn, qp, kv, nb, bs, bt, mb, sl, _ptr(idx),
                                            idx.shape[1], sc, _ptr(out), _ptr(lse),
                                            int(n_threads),
                                            _ptr(f8) if f8 is not None else None,
                                            float(kv_scale)), "oracle_mla_decode_sparse")
    del keep
    return out, lse


def e4m3_decode(codes):
    """OCP E4M3 bytes (any shape, uint8) -> float64 values of the same shape."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape, dtype=np.float64)
    _check(_load().oracle_e4m3_decode(codes.size, _ptr(codes), _ptr(out)), "oracle_e4m3_decode")
    return out


def mla_decode_fp8(q_nope, q_pe, kv_fp8, kv_scale, block_table, seq_lens, sm_scale,
                   n_threads: int = 0):
    """Decode over an FP8 latent cache: kv_fp8 uint8 [num_blocks, bs, 576] of
    E4M3 bytes, element value kv_scale * e4m3(byte). q_nope [B, H, 512] (or
    [B, q_len, H, 512] for multi-token queries, causal as in mla_decode_multi).
    Returns (out, lse) shaped like the queries without the last axis / with 512."""
    q_nope = np.ascontiguousarray(q_nope, dtype=np.uint16)
    q_pe = np.ascontiguousarray(q_pe, dtype=np.uint16)
    multi = q_nope.ndim == 4
    if multi:
        B, q_len, H, dc = q_nope.shape
    else:
        (B, H, dc), q_len = q_nope.shape, 1
    assert dc == D_C and q_pe.shape == q_nope.shape[:-1] + (D_R,), (q_nope.shape, q_pe.shape)
    kv_fp8 = np.ascontiguousarray(kv_fp8, dtype=np.uint8)
    nb, bs, d = kv_fp8.shape
    assert d == D, kv_fp8.shape
    block_table = np.ascontiguousarray(block_table, dtype=np.int32)
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    assert block_table.ndim == 2 and block_table.shape[0] == B and seq_lens.shape == (B,)
    out = np.empty(q_nope.shape[:-1] + (D_C,), dtype=np.float64)
    lse = np.empty(q_nope.shape[:-1], dtype=np.float64)
    _check(_load().oracle_mla_decode_fp8(B, q_len, H, _ptr(q_nope), _ptr(q_pe), _ptr(kv_fp8),
                                         float(kv_scale), nb, bs, _ptr(block_table),
                                         block_table.shape[1], _ptr(seq_lens), float(sm_scale),
                                         _ptr(out), _ptr(lse), int(n_threads)),
           "oracle_mla_decode_fp8")
    return out, lse


def mla_decode_rows(q_nope, q_pe, kv_cache, block_table, seq_lens, sm_scale, rows_b, rows_h,
                    n_threads: int = 0):
    """Decode only the listed (b, h) rows: returns (out[n, 512], lse[n])."""
    args, keep = _common(q_nope, q_pe, kv_cache, block_table, seq_lens, sm_scale)
    rb = np.ascontiguousarray(rows_b, dtype=np.int32)
    rh = np.ascontiguousarray(rows_h, dtype=np.int32)
    assert rb.shape == rh.shape and rb.ndim == 1
    n = rb.shape[0]
    out = np.empty((n, D_C), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    _check(_load().oracle_mla_decode_rows(*args, n, _ptr(rb), _ptr(rh), _ptr(out), _ptr(lse),
                                          int(n_threads)), "oracle_mla_decode_rows")
    del keep
    return out, lse


def mla_partial(q_nope, q_pe, kv_cache, block_table, seq_lens, sm_scale, b, h, t0, t1):
    """Split-KV partial of (b, h) over tokens [t0, t1): (o[512], lse)."""
    args, keep = _common(q_nope, q_pe, kv_cache, block_table, seq_lens, sm_scale)
    o = np.empty((D_C,), dtype=np.float64)
    lse = np.empty((1,), dtype=np.float64)
    _check(_load().oracle_mla_partial(*args, int(b), int(h), int(t0), int(t1), _ptr(o),
                                      _ptr(lse)), "oracle_mla_partial")
    del keep
    return o, float(lse[0])


def mla_combine(o_parts, lse_parts):
    """Merge split partials o_parts[n, 512], lse_parts[n] -> (o[512], lse)."""
    o_parts = np.ascontiguousarray(o_parts, dtype=np.float64).reshape(-1, D_C)
    lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64).reshape(-1)
    assert o_parts.shape[0] == lse_parts.shape[0]
    o = np.empty((D_C,), dtype=np.float64)
    lse = np.empty((1,), dtype=np.float64)
    _check(_load().oracle_mla_combine(o_parts.shape[0], _ptr(o_parts), _ptr(lse_parts), _ptr(o),
                                      _ptr(lse)), "oracle_mla_combine")
    return o, float(lse[0])


def mla_decode_bruteforce(q_nope, q_pe, kv_cache, block_table, seq_lens, sm_scale):
    """Independent long-double path for tiny inputs: (out, lse) as float64."""
    args, keep = _common(q_nope, q_pe, kv_cache, block_table, seq_lens, sm_scale)
    B, H = args[0], args[1]
    out = np.empty((B, H, D_C), dtype=np.float64)
    lse = np.empty((B, H), dtype=np.float64)
    _check(_load().oracle_mla_decode_bruteforce(*args, _ptr(out), _ptr(lse)),
           "oracle_mla_decode_bruteforce")
    del keep
    return out, lse
