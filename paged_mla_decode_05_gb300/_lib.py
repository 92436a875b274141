"""ctypes binding of ``include/mla_decode.h``: same names, argument marshalling only.

Every step of the decode runs in the sm_103a kernels of the shared library;
this module converts torch tensors to pointers, checks dtypes, shapes and
devices, and turns status codes into exceptions. There is no fallback: if the
library is missing the import of this module fails.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import List, Optional, Tuple

import numpy as np

from . import build as _build

D_C = 512
D_R = 64
D = D_C + D_R
HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "mla_decode.h")

MLA_OK = 0
STATUS_NAMES = {0: "MLA_OK", 1: "MLA_ERR_INVALID_ARG", 2: "MLA_ERR_UNSUPPORTED_DEVICE",
                3: "MLA_ERR_WORKSPACE_TOO_SMALL", 4: "MLA_ERR_CUDA", 5: "MLA_ERR_DEVICE_FAULT"}
MLA_DEVERR_BAD_BLOCK = 1
MLA_DEVERR_SEQLEN_MISMATCH = 2
MLA_DEVERR_TIMEOUT = 4


class MLAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")


class PlanOptions(ctypes.Structure):
    _fields_ = [("num_clusters", ctypes.c_int), ("force_splits", ctypes.c_int),
                ("host_only", ctypes.c_int), ("lengths_are_bounds", ctypes.c_int),
                ("q_len", ctypes.c_int)]


def _load() -> ctypes.CDLL:
    path = _build.LIB_PATH
    if not os.path.exists(path):
        raise ImportError(f"paged MLA decode library not built ({path}); run "
                          "`python -m paged_mla_decode_05_gb300.build` (needs nvcc)")
    lib = ctypes.CDLL(path)
    p, i32, i64, u32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint32
    sz = ctypes.c_size_t
    sigs = {
        "mla_decode_plan": (i32, [i32, i32, p, i32, i32, p]),
        "mla_decode_plan_ex": (i32, [i32, i32, p, i32, i32, ctypes.POINTER(PlanOptions), p]),
        "mla_plan_update": (i32, [p, p, p]),
        "mla_plan_workspace_bytes": (sz, [p]),
        "mla_plan_num_splits": (i32, [p, i32]),
        "mla_plan_num_work_items": (i32, [p]),
        "mla_plan_num_clusters": (i32, [p]),
        "mla_plan_work_item": (i32, [p, i32, p, p, p, p, p]),
        "mla_plan_work_item_heads": (i32, [p, i32, p, p]),
        "mla_decode": (i32, [p, p, p, p, i64, p, p, ctypes.c_float, p, p, p, sz, p]),
        "mla_decode_fp8": (i32, [p, p, p, p, ctypes.c_float, i64, p, p, ctypes.c_float, p, p, p,
                                 sz, p]),
        "mla_decode_no_alloc": (i32, [p, p, p, p, i64, p, p, ctypes.c_float, p, p, p, p]),
        "mla_sparse_plan": (i32, [i32, i32, i32, ctypes.POINTER(PlanOptions), p]),
        "mla_decode_sparse": (i32, [p, p, p, p, i32, ctypes.c_float, i64, i32, p, i32, p, p,
                                    ctypes.c_float, p, p, p, sz, p]),
        "mla_check_device_error": (i32, [p, p, ctypes.POINTER(u32)]),
        "mla_plan_destroy": (None, [p]),
        "mla_status_string": (ctypes.c_char_p, [i32]),
        "mla_device_supported": (i32, []),
        "mla_selftest_wait_timeout": (i32, [p, ctypes.POINTER(u32)]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


LIB = _load()


def header_functions() -> List[str]:
    """Names of the functions declared in include/mla_decode.h."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z_0-9]+)\s*\(", text)))


def _check(status: int, what: str):
    if status != MLA_OK:
        raise MLAError(status, what)


def mla_device_supported() -> bool:
    return bool(LIB.mla_device_supported())


class Plan:
    """Owns an ``mla_plan_t``; freed on ``destroy()`` or garbage collection."""

    def __init__(self, handle: int, B: int, H: int, block_size: int, max_blocks: int,
                 host_only: bool, q_len: int = 1):
        self._h = ctypes.c_void_p(handle)
        self.B, self.H, self.block_size, self.max_blocks = B, H, block_size, max_blocks
        self.host_only = host_only
        self.q_len = q_len

    def q_shape(self, d: int):
        """Shape of a per-query-row tensor with trailing dimension d (None: none)."""
        lead = (self.B, self.H) if self.q_len == 1 else (self.B, self.q_len, self.H)
        return lead if d is None else lead + (d,)

    @property
    def handle(self) -> ctypes.c_void_p:
        if not self._h:
            raise ValueError("plan destroyed")
        return self._h

    def destroy(self):
        if self._h:
            LIB.mla_plan_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass

    @property
    def workspace_bytes(self) -> int:
        return int(LIB.mla_plan_workspace_bytes(self.handle))

    def num_splits(self, b: int) -> int:
        return int(LIB.mla_plan_num_splits(self.handle, b))

    @property
    def num_work_items(self) -> int:
        return int(LIB.mla_plan_num_work_items(self.handle))

    @property
    def num_clusters(self) -> int:
        return int(LIB.mla_plan_num_clusters(self.handle))

    def work_items(self) -> List[Tuple[int, int, int, int, int]]:
        out = []
        vals = [ctypes.c_int32() for _ in range(5)]
        for i in range(self.num_work_items):
            rc = LIB.mla_plan_work_item(self.handle, i, *(ctypes.byref(v) for v in vals))
            if rc != 0:
                raise MLAError(MLA_OK + 1, "mla_plan_work_item")
            out.append(tuple(v.value for v in vals))
        return out

    def work_item_heads(self) -> List[Tuple[int, int]]:
        """Query heads [h_begin, h_end) of every work item (its head group)."""
        out = []
        hb, he = ctypes.c_int32(), ctypes.c_int32()
        for i in range(self.num_work_items):
            rc = LIB.mla_plan_work_item_heads(self.handle, i, ctypes.byref(hb), ctypes.byref(he))
            if rc != 0:
                raise MLAError(MLA_OK + 1, "mla_plan_work_item_heads")
            out.append((hb.value, he.value))
        return out

    def update(self, seq_lens_host, stream=None):
        lens = np.ascontiguousarray(np.asarray(seq_lens_host, dtype=np.int32))
        if lens.shape != (self.B,):
            raise ValueError(f"seq_lens must have shape ({self.B},)")
        _check(LIB.mla_plan_update(self.handle, lens.ctypes.data_as(ctypes.c_void_p),
                                   _stream_ptr(stream)), "mla_plan_update")


def mla_decode_plan(B: int, H: int, seq_lens_host, block_size: int, max_blocks: int,
                    num_clusters: int = 0, force_splits: int = 0, host_only: bool = False,
                    lengths_are_bounds: bool = False, q_len: int = 1) -> Plan:
    """Build the split-KV schedule (host-only; uploads a small work list).

    With ``lengths_are_bounds`` the host lengths are upper bounds and every
    decode reads the true lengths from the device ``seq_lens`` (a launch that
    can be captured once in a CUDA graph and replayed as lengths change).
    ``q_len`` > 1: several query tokens per request (speculative decoding);
    query tensors and outputs then take the shape [B, q_len, H, ...]."""
    lens = np.ascontiguousarray(np.asarray(seq_lens_host, dtype=np.int32))
    if lens.shape != (B,):
        raise ValueError(f"seq_lens must have shape ({B},)")
    opts = PlanOptions(int(num_clusters), int(force_splits), 1 if host_only else 0,
                       1 if lengths_are_bounds else 0, int(q_len))
    h = ctypes.c_void_p()
    _check(LIB.mla_decode_plan_ex(B, H, lens.ctypes.data_as(ctypes.c_void_p), block_size,
                                  max_blocks, ctypes.byref(opts), ctypes.byref(h)),
           "mla_decode_plan")
    return Plan(h.value, B, H, block_size, max_blocks, host_only, int(q_len))


def mla_sparse_plan(B: int, H: int, topk: int, num_clusters: int = 0, force_splits: int = 0,
                    host_only: bool = False) -> Plan:
    """Plan a sparse (top-k) decode: B requests of H heads, topk list entries
    each (see mla_sparse_plan in include/mla_decode.h). The plan serves any
    lists and lengths."""
    opts = PlanOptions(int(num_clusters), int(force_splits), 1 if host_only else 0, 1, 1)
    h = ctypes.c_void_p()
    _check(LIB.mla_sparse_plan(B, H, int(topk), ctypes.byref(opts), ctypes.byref(h)),
           "mla_sparse_plan")
    plan = Plan(h.value, B, H, 64, -(-int(topk) // 64), host_only, 1)
    plan.topk = int(topk)
    return plan


def mla_decode_sparse(plan: Plan, q_nope, q_pe, kv_cache, block_table, seq_lens, topk_indices,
                      sm_scale: float, out, lse, workspace, kv_scale: float = None, stream=None):
    """Enqueue one sparse decode (see mla_decode_sparse in include/mla_decode.h).

    kv_cache: bf16 [num_blocks, block_size, 576], or uint8 / float8_e4m3fn
    E4M3 bytes with ``kv_scale``; block_table int32 [B, max_blocks]; seq_lens
    int32 [B]; topk_indices int32 [B, topk]; workspace a CUDA uint8 tensor of
    at least plan.workspace_bytes bytes."""
    import torch
    topk = getattr(plan, "topk", None)
    if topk is None:
        raise ValueError("plan was not made by mla_sparse_plan")
    B, H = plan.B, plan.H
    f8 = getattr(torch, "float8_e4m3fn", None)
    if f8 is not None and kv_cache.dtype == f8:
        kv_cache = kv_cache.view(torch.uint8)
    fp8 = kv_cache.dtype == torch.uint8
    if fp8 != (kv_scale is not None):
        raise ValueError("an FP8 cache needs kv_scale; a bf16 cache takes none")
    if kv_cache.dim() != 3 or kv_cache.shape[2] != D:
        raise ValueError(f"kv_cache must have shape [num_blocks, block_size, {D}]")
    nb, bs = int(kv_cache.shape[0]), int(kv_cache.shape[1])
    kv = _tensor(kv_cache, torch.uint8 if fp8 else torch.bfloat16, (nb, bs, D), "kv_cache")
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError(f"block_table must have shape [{B}, max_blocks]")
    mb = int(block_table.shape[1])
    bt = _tensor(block_table, torch.int32, (B, mb), "block_table")
    sl = _tensor(seq_lens, torch.int32, (B,), "seq_lens")
    ti = _tensor(topk_indices, torch.int32, (B, topk), "topk_indices")
    qn = _tensor(q_nope, torch.bfloat16, (B, H, D_C), "q_nope")
    qp = _tensor(q_pe, torch.bfloat16, (B, H, D_R), "q_pe")
    o = _tensor(out, torch.bfloat16, (B, H, D_C), "out")
    l = _tensor(lse, torch.float32, (B, H), "lse")
    if workspace is None or not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(LIB.mla_decode_sparse(plan.handle, qn, qp, kv, 1 if fp8 else 0,
                                 ctypes.c_float(kv_scale if fp8 else 1.0), nb, bs, bt, mb, sl, ti,
                                 ctypes.c_float(sm_scale), o, l,
                                 ctypes.c_void_p(workspace.data_ptr()), ws_bytes,
                                 _stream_ptr(stream)), "mla_decode_sparse")


def _stream_ptr(stream) -> ctypes.c_void_p:
    if stream is None:
        import torch
        if not torch.cuda.is_available():
            return ctypes.c_void_p(0)
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _tensor(t, dtype, shape, name):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def mla_decode(plan: Plan, q_nope, q_pe, kv_cache, block_table, seq_lens, sm_scale: float, out,
               lse, workspace=None, stream=None):
    """Enqueue one decode (see mla_decode in include/mla_decode.h).

    Tensors: q_nope bf16 [B,H,512], q_pe bf16 [B,H,64], kv_cache bf16
    [num_blocks, block_size, 576], block_table int32 [B, max_blocks], seq_lens
    int32 [B] (all CUDA); out bf16 [B,H,512] and lse fp32 [B,H] are written;
    workspace is a CUDA uint8 tensor of at least plan.workspace_bytes bytes.
    """
    import torch
    B, H = plan.B, plan.H
    if kv_cache.dim() != 3 or kv_cache.shape[1] != plan.block_size or kv_cache.shape[2] != D:
        raise ValueError(f"kv_cache must have shape [num_blocks, {plan.block_size}, {D}]")
    nb = int(kv_cache.shape[0])
    args = [
        _tensor(q_nope, torch.bfloat16, plan.q_shape(D_C), "q_nope"),
        _tensor(q_pe, torch.bfloat16, plan.q_shape(D_R), "q_pe"),
        _tensor(kv_cache, torch.bfloat16, (nb, plan.block_size, D), "kv_cache"),
    ]
    bt = _tensor(block_table, torch.int32, (B, plan.max_blocks), "block_table")
    sl = _tensor(seq_lens, torch.int32, (B,), "seq_lens")
    o = _tensor(out, torch.bfloat16, plan.q_shape(D_C), "out")
    l = _tensor(lse, torch.float32, plan.q_shape(None), "lse")
    if workspace is None:
        ws, ws_bytes = ctypes.c_void_p(0), 0
    else:
        if not workspace.is_cuda or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous CUDA tensor")
        ws = ctypes.c_void_p(workspace.data_ptr())
        ws_bytes = workspace.numel() * workspace.element_size()
    _check(LIB.mla_decode(plan.handle, args[0], args[1], args[2], nb, bt, sl,
                          ctypes.c_float(sm_scale), o, l, ws, ws_bytes, _stream_ptr(stream)),
           "mla_decode")


def mla_decode_fp8(plan: Plan, q_nope, q_pe, kv_cache_fp8, kv_scale: float, block_table,
                   seq_lens, sm_scale: float, out, lse, workspace=None, stream=None):
    """Enqueue one decode over an FP8 (E4M3) latent cache (see mla_decode_fp8
    in include/mla_decode.h).

    kv_cache_fp8 is a CUDA uint8 tensor [num_blocks, block_size, 576] of E4M3
    bytes (a float8_e4m3fn tensor viewed as uint8 is accepted too); element
    values are kv_scale * e4m3(byte). Everything else as ``mla_decode``.
    """
    import torch
    B, H = plan.B, plan.H
    if getattr(torch, "float8_e4m3fn", None) is not None and kv_cache_fp8.dtype == torch.float8_e4m3fn:
        kv_cache_fp8 = kv_cache_fp8.view(torch.uint8)
    if (kv_cache_fp8.dim() != 3 or kv_cache_fp8.shape[1] != plan.block_size
            or kv_cache_fp8.shape[2] != D):
        raise ValueError(f"kv_cache_fp8 must have shape [num_blocks, {plan.block_size}, {D}]")
    nb = int(kv_cache_fp8.shape[0])
    args = [
        _tensor(q_nope, torch.bfloat16, plan.q_shape(D_C), "q_nope"),
        _tensor(q_pe, torch.bfloat16, plan.q_shape(D_R), "q_pe"),
        _tensor(kv_cache_fp8, torch.uint8, (nb, plan.block_size, D), "kv_cache_fp8"),
    ]
    bt = _tensor(block_table, torch.int32, (B, plan.max_blocks), "block_table")
    sl = _tensor(seq_lens, torch.int32, (B,), "seq_lens")
    o = _tensor(out, torch.bfloat16, plan.q_shape(D_C), "out")
    l = _tensor(lse, torch.float32, plan.q_shape(None), "lse")
    if workspace is None:
        ws, ws_bytes = ctypes.c_void_p(0), 0
    else:
        if not workspace.is_cuda or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous CUDA tensor")
        ws = ctypes.c_void_p(workspace.data_ptr())
        ws_bytes = workspace.numel() * workspace.element_size()
    _check(LIB.mla_decode_fp8(plan.handle, args[0], args[1], args[2], ctypes.c_float(kv_scale), nb,
                              bt, sl, ctypes.c_float(sm_scale), o, l, ws, ws_bytes,
                              _stream_ptr(stream)),
           "mla_decode_fp8")


def mla_decode_no_alloc(plan: Plan, q_nope, q_pe, kv_cache, block_table, seq_lens,
                        sm_scale: float, out, lse, err_bits, stream=None):
    """Enqueue one decode that allocates nothing (see mla_decode_no_alloc in
    include/mla_decode.h): for callers whose device memory all belongs to a
    caching allocator, or who must not stall on cudaMalloc's synchronisation.

    Same tensors as ``mla_decode`` but no workspace: the split partials live in
    the library's fixed device scratch, shared by every call on the device, so
    calls that may overlap on the GPU race. ``plan`` may be host-only.
    ``err_bits`` is a CUDA int32 tensor of one element that receives this
    call's device error bits. A stream under graph capture is refused.
    """
    import torch
    B, H = plan.B, plan.H
    if kv_cache.dim() != 3 or kv_cache.shape[1] != plan.block_size or kv_cache.shape[2] != D:
        raise ValueError(f"kv_cache must have shape [num_blocks, {plan.block_size}, {D}]")
    nb = int(kv_cache.shape[0])
    args = [
        _tensor(q_nope, torch.bfloat16, plan.q_shape(D_C), "q_nope"),
        _tensor(q_pe, torch.bfloat16, plan.q_shape(D_R), "q_pe"),
        _tensor(kv_cache, torch.bfloat16, (nb, plan.block_size, D), "kv_cache"),
    ]
    bt = _tensor(block_table, torch.int32, (B, plan.max_blocks), "block_table")
    sl = _tensor(seq_lens, torch.int32, (B,), "seq_lens")
    o = _tensor(out, torch.bfloat16, plan.q_shape(D_C), "out")
    l = _tensor(lse, torch.float32, plan.q_shape(None), "lse")
    eb = _tensor(err_bits, torch.int32, (1,), "err_bits")
    _check(LIB.mla_decode_no_alloc(plan.handle, args[0], args[1], args[2], nb, bt, sl,
                                   ctypes.c_float(sm_scale), o, l, eb, _stream_ptr(stream)),
           "mla_decode_no_alloc")


def mla_check_device_error(plan: Plan, stream=None) -> int:
    """Synchronise, read and clear the plan's device error bits (0 = none)."""
    bits = ctypes.c_uint32(0)
    st = LIB.mla_check_device_error(plan.handle, _stream_ptr(stream), ctypes.byref(bits))
    if st not in (MLA_OK, 5):
        raise MLAError(st, "mla_check_device_error")
    return int(bits.value)


def mla_selftest_wait_timeout(stream=None) -> int:
    """Run the bounded-wait health check (about a second on the current device)
    and return the MLA_DEVERR_* bits it produced: MLA_DEVERR_TIMEOUT when the
    wait gave up as designed."""
    bits = ctypes.c_uint32(0)
    _check(LIB.mla_selftest_wait_timeout(_stream_ptr(stream), ctypes.byref(bits)),
           "mla_selftest_wait_timeout")
    return int(bits.value)


def mla_status_string(status: int) -> str:
    return LIB.mla_status_string(int(status)).decode()
