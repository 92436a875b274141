"""Convenience wrapper: allocate outputs and workspace, plan, decode."""
from __future__ import annotations

from ._lib import Plan, mla_decode, mla_decode_fp8, mla_decode_plan


def decode(q_nope, q_pe, kv_cache, block_table, seq_lens, sm_scale: float, seq_lens_host=None,
           plan: Plan = None, stream=None, kv_scale: float = None):
    """One decode step on torch CUDA tensors; returns (out bf16 [B,H,512], lse fp32 [B,H]).

    ``seq_lens_host`` (host int array) is needed to plan unless ``plan`` is given.
    A uint8 (or float8_e4m3fn) ``kv_cache`` is an FP8 E4M3 cache and needs
    ``kv_scale``; a bf16 one must not be given a scale.
    """
    import torch
    B, H, _ = q_nope.shape
    fp8 = kv_cache.dtype == torch.uint8 or kv_cache.dtype == getattr(torch, "float8_e4m3fn", None)
    if fp8 != (kv_scale is not None):
        raise ValueError("an FP8 cache needs kv_scale; a bf16 cache takes none")
    if plan is None:
        if seq_lens_host is None:
            seq_lens_host = seq_lens.cpu().numpy()
        plan = mla_decode_plan(B, H, seq_lens_host, int(kv_cache.shape[1]),
                               int(block_table.shape[1]))
    out = torch.empty((B, H, 512), dtype=torch.bfloat16, device=q_nope.device)
    lse = torch.empty((B, H), dtype=torch.float32, device=q_nope.device)
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
