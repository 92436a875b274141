"""Convenience wrappers: allocate outputs and workspace, plan, decode."""
from __future__ import annotations

from ._lib import (Plan, mla_decode, mla_decode_fp8, mla_decode_plan, mla_decode_sparse,
                   mla_sparse_plan)


def _is_fp8(kv_cache, kv_scale):
    import torch
    fp8 = kv_cache.dtype == torch.uint8 or kv_cache.dtype == getattr(torch, "float8_e4m3fn", None)
    if fp8 != (kv_scale is not None):
        raise ValueError("an FP8 cache needs kv_scale; a bf16 cache takes none")
    return fp8


def decode(q_nope, q_pe, kv_cache, block_table, seq_lens, sm_scale: float, seq_lens_host=None,
           plan: Plan = None, stream=None, kv_scale: float = None):
    """One decode step on torch CUDA tensors; returns (out bf16, lse fp32).

    q_nope is [B, H, 512], or [B, q_len, H, 512] for q_len query tokens per
    request (speculative decoding: token j sees the request's first
    L - q_len + 1 + j tokens); out and lse take the queries' shape.
    ``seq_lens_host`` (host int array) is needed to plan unless ``plan`` is given.
    A uint8 (or float8_e4m3fn) ``kv_cache`` is an FP8 E4M3 cache and needs
    ``kv_scale``; a bf16 one must not be given a scale.
    """
    import torch
    if q_nope.dim() == 4:
        B, q_len, H, _ = q_nope.shape
    else:
        (B, H, _), q_len = q_nope.shape, 1
    fp8 = _is_fp8(kv_cache, kv_scale)
    if plan is None:
        if seq_lens_host is None:
            seq_lens_host = seq_lens.cpu().numpy()
        plan = mla_decode_plan(B, H, seq_lens_host, int(kv_cache.shape[1]),
                               int(block_table.shape[1]), q_len=q_len)
    out = torch.empty(plan.q_shape(512), dtype=torch.bfloat16, device=q_nope.device)
    lse = torch.empty(plan.q_shape(None), dtype=torch.float32, device=q_nope.device)
    ws = None
    if plan.workspace_bytes:
        ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=q_nope.device)
    if fp8:
        mla_decode_fp8(plan, q_nope, q_pe, kv_cache, kv_scale, block_table, seq_lens, sm_scale,
                       out, lse, ws, stream)
    else:
        mla_decode(plan, q_nope, q_pe, kv_cache, block_table, seq_lens, sm_scale, out, lse, ws,
                   stream)
    return out, lse


def decode_sparse(q_nope, q_pe, kv_cache, block_table, seq_lens, topk_indices, sm_scale: float,
                  plan: Plan = None, stream=None, kv_scale: float = None):
    """One sparse (top-k) decode step: request b attends to the tokens listed
    in topk_indices[b] (int32 [B, topk]; entries outside [0, L) are padding).
    Returns (out bf16 [B, H, 512], lse fp32 [B, H]). A plan from
    mla_sparse_plan(B, H, topk) may be passed to reuse it across steps."""
    import torch
    B, H, _ = q_nope.shape
    fp8 = _is_fp8(kv_cache, kv_scale)
    if plan is None:
        plan = mla_sparse_plan(B, H, int(topk_indices.shape[1]))
    out = torch.empty((B, H, 512), dtype=torch.bfloat16, device=q_nope.device)
    lse = torch.empty((B, H), dtype=torch.float32, device=q_nope.device)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=q_nope.device)
    mla_decode_sparse(plan, q_nope, q_pe, kv_cache, block_table, seq_lens, topk_indices, sm_scale,
                      out, lse, ws, kv_scale=kv_scale if fp8 else None, stream=stream)
    return out, lse
