"""GB300 (sm_103a) causal multi-head attention: forward and its VJP, and paged
decode attention (one query token per request over a paged K/V cache).

The computation lives in librca_attn.so (hand-written CUDA, C ABI in
include/rca_attn.h). This package only allocates outputs with torch and
marshals pointers; there is no CPU or library fallback.
"""

from __future__ import annotations

from . import _native
from ._native import (  # noqa: F401  (C-ABI names)
    RcaError,
    rca_abi_version,
    rca_attn_bwd,
    rca_attn_bwd_dq_convert,
    rca_attn_bwd_main,
    rca_attn_bwd_noalloc,
    rca_attn_bwd_preprocess,
    rca_attn_bwd_qkv,
    rca_attn_bwd_varlen,
    rca_attn_bwd_workspace_size,
    rca_attn_fwd,
    rca_attn_fwd_qkv,
    rca_attn_fwd_varlen,
    rca_attn_materialized_bwd,
    rca_attn_varlen_workspace_size,
    rca_attn_materialized_fwd,
    rca_attn_materialized_workspace_size,
    rca_causal_softmax,
    rca_causal_softmax_bwd,
    rca_causal_softmax_bwd_tiled,
    rca_last_error,
    rca_paged_decode,
    rca_paged_decode_workspace_size,
    rca_selftest_device_timeout,
    rca_selftest_noalloc_timeout,
    rca_set_wait_timeout_ns,
    rca_stream_status,
)

__all__ = [
    "attention_forward",
    "attention_backward",
    "CausalAttention",
    "causal_attention",
    "RcaError",
    "rca_abi_version",
    "rca_attn_fwd",
    "rca_attn_bwd",
    "rca_attn_bwd_workspace_size",
    "rca_attn_bwd_preprocess",
    "rca_attn_bwd_main",
    "rca_attn_bwd_dq_convert",
    "rca_attn_bwd_noalloc",
    "attention_forward_qkv",
    "attention_backward_qkv",
    "causal_attention_qkv",
    "rca_attn_fwd_qkv",
    "rca_attn_bwd_qkv",
    "attention_forward_varlen",
    "attention_backward_varlen",
    "rca_attn_fwd_varlen",
    "rca_attn_bwd_varlen",
    "rca_attn_varlen_workspace_size",
    "materialized_forward",
    "materialized_backward",
    "rca_attn_materialized_fwd",
    "rca_attn_materialized_bwd",
    "rca_attn_materialized_workspace_size",
    "rca_causal_softmax",
    "rca_causal_softmax_bwd",
    "rca_causal_softmax_bwd_tiled",
    "paged_decode",
    "rca_paged_decode",
    "rca_paged_decode_workspace_size",
    "rca_stream_status",
    "rca_last_error",
    "rca_set_wait_timeout_ns",
    "rca_selftest_device_timeout",
    "rca_selftest_noalloc_timeout",
]


def attention_forward(q, k, v, stream=None):
    """Returns (out [B,T,Hq,Dh] in q's dtype, lse [B,Hq,T] float32)."""
    import torch

    B, T, Hq, Dh = q.shape
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq, T), dtype=torch.float32, device=q.device)
    rca_attn_fwd(q, k, v, out, lse, stream)
    return out, lse


def workspace_for(q, k):
    """Device scratch for the backward of these q [B,T,Hq,Dh] / k [B,T,Hkv,Dh]."""
    import torch

    B, T, Hq, Dh = q.shape
    n = rca_attn_bwd_workspace_size(B, Hq, k.shape[2], T, Dh, q.dtype)
    return torch.empty(n, dtype=torch.uint8, device=q.device)


def attention_backward(q, k, v, out, lse, dout, workspace=None, stream=None):
    """Returns (dq, dk, dv) in the storage dtype."""
    import torch

    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    ws = workspace if workspace is not None else workspace_for(q, k)
    rca_attn_bwd(q, k, v, out, lse, dout.contiguous(), dq, dk, dv, ws, stream)
    return dq, dk, dv


def materialized_workspace_for(q, k):
    import torch

    B, T, Hq, Dh = q.shape
    n = rca_attn_materialized_workspace_size(B, Hq, k.shape[2], T, Dh, q.dtype)
    return torch.empty(n, dtype=torch.uint8, device=q.device)


def materialized_forward(q, k, v, workspace=None, stream=None):
    """Materialized path / probability-returning diagnostic. Returns (out
    [B,T,Hq,Dh] in q's dtype, probs [B,Hq,T,T] float32, lse [B,Hq,T] float32)."""
    import torch

    B, T, Hq, Dh = q.shape
    out = torch.empty_like(q)
    probs = torch.empty((B, Hq, T, T), dtype=torch.float32, device=q.device)
    lse = torch.empty((B, Hq, T), dtype=torch.float32, device=q.device)
    ws = workspace if workspace is not None else materialized_workspace_for(q, k)
    rca_attn_materialized_fwd(q, k, v, out, probs, lse, ws, stream)
    return out, probs, lse


def materialized_backward(q, k, v, probs, dout, dprobs=None, workspace=None, stream=None):
    """VJP of (out, probs) from the stored probabilities. Returns (dq, dk, dv)."""
    import torch

    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    ws = workspace if workspace is not None else materialized_workspace_for(q, k)
    rca_attn_materialized_bwd(q, k, v, probs, dout.contiguous(), dprobs, dq, dk, dv, ws, stream)
    return dq, dk, dv


def paged_decode(q, k_pool, v_pool, page_table, seq_lens, workspace=None, stream=None):
    """One decode step: q [B,Hq,Dh] over pools [P,Hkv,page_size,Dh] through
    page_table [B,max_pages] (int32) for seq_lens [B] (int32) cached positions.
    Returns (out [B,Hq,Dh] in q's dtype, lse [B,Hq] float32). Inference only."""
    import torch

    B, Hq, Dh = q.shape
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        n = rca_paged_decode_workspace_size(B, Hq, k_pool.shape[1], Dh, k_pool.shape[2], page_table.shape[1],
                                            q.dtype)
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)
    rca_paged_decode(q, k_pool, v_pool, page_table, seq_lens, out, lse, workspace, stream)
    return out, lse


def varlen_workspace_for(q, k):
    import torch

    B, T, Hq, Dh = q.shape
    n = rca_attn_varlen_workspace_size(B, Hq, k.shape[2], T, Dh, q.dtype)
    return torch.empty(n, dtype=torch.uint8, device=q.device)


def attention_forward_varlen(q, k, v, seq_lens, workspace=None, stream=None):
    """Right-padded batch with per-sequence lengths seq_lens (int32 [B], device).
    Returns (out, lse); padding rows are zero, their LSE -inf."""
    import torch

    B, T, Hq, Dh = q.shape
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq, T), dtype=torch.float32, device=q.device)
    ws = workspace if workspace is not None else varlen_workspace_for(q, k)
    rca_attn_fwd_varlen(q, k, v, seq_lens, out, lse, ws, stream)
    return out, lse


def attention_backward_varlen(q, k, v, out, lse, dout, seq_lens, workspace=None, stream=None):
    """Returns (dq, dk, dv); zero at padding positions, dout there is ignored."""
    import torch

    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = workspace if workspace is not None else varlen_workspace_for(q, k)
    rca_attn_bwd_varlen(q, k, v, out, lse, dout.contiguous(), seq_lens, dq, dk, dv, ws, stream)
    return dq, dk, dv


def attention_forward_qkv(qkv, Hq, Hkv, stream=None):
    """Fused layout: qkv [B,T,(Hq+2*Hkv)*Dh] -> (out [B,T,Hq*Dh], lse [B,Hq,T])."""
    import torch

    B, T, W = qkv.shape
    Dh = W // (Hq + 2 * Hkv)
    out = torch.empty((B, T, Hq * Dh), dtype=qkv.dtype, device=qkv.device)
    lse = torch.empty((B, Hq, T), dtype=torch.float32, device=qkv.device)
    rca_attn_fwd_qkv(qkv, Hq, Hkv, out, lse, stream)
    return out, lse


def attention_backward_qkv(qkv, Hq, Hkv, out, lse, dout, workspace=None, stream=None):
    """Returns dqkv [B,T,(Hq+2*Hkv)*Dh] (the gradient of the fused projection output)."""
    import torch

    B, T, W = qkv.shape
    Dh = W // (Hq + 2 * Hkv)
    dqkv = torch.empty_like(qkv)
    if workspace is None:
        n = rca_attn_bwd_workspace_size(B, Hq, Hkv, T, Dh, qkv.dtype)
        workspace = torch.empty(n, dtype=torch.uint8, device=qkv.device)
    rca_attn_bwd_qkv(qkv, Hq, Hkv, out, lse, dout.contiguous(), dqkv, workspace, stream)
    return dqkv


def _autograd_qkv_cls():
    import torch

    class CausalAttentionQKV(torch.autograd.Function):
        """Custom-gradient node over the fused layout: input qkv, output the
        merged heads; the VJP returns the gradient of qkv in the same layout."""

        @staticmethod
        def forward(ctx, qkv, Hq, Hkv):
            out, lse = attention_forward_qkv(qkv, Hq, Hkv)
            ctx.save_for_backward(qkv, out, lse)
            ctx.heads = (Hq, Hkv)
            return out

        @staticmethod
        def backward(ctx, dout):
            qkv, out, lse = ctx.saved_tensors
            return attention_backward_qkv(qkv, *ctx.heads, out, lse, dout), None, None

    return CausalAttentionQKV


def causal_attention_qkv(qkv, Hq, Hkv):
    """Differentiable causal attention on a fused projection output
    [B,T,(Hq+2*Hkv)*Dh]; returns [B,T,Hq*Dh] for the output projection."""
    if _Lazy.qkv_cls is None:
        _Lazy.qkv_cls = _autograd_qkv_cls()
    return _Lazy.qkv_cls.apply(qkv, Hq, Hkv)


def _autograd_cls():
    import torch

    class CausalAttention(torch.autograd.Function):
        """torch.autograd wrapper: saves q, k, v, out and lse; backward recomputes P."""

        @staticmethod
        def forward(ctx, q, k, v):
            out, lse = attention_forward(q, k, v)
            ctx.save_for_backward(q, k, v, out, lse)
            return out

        @staticmethod
        def backward(ctx, dout):
            q, k, v, out, lse = ctx.saved_tensors
            return attention_backward(q, k, v, out, lse, dout)

    return CausalAttention


class _Lazy:
    cls = None
    qkv_cls = None


def causal_attention(q, k, v):
    """Differentiable causal attention over [B,T,H,Dh] tensors (GQA when Hkv < Hq)."""
    if _Lazy.cls is None:
        _Lazy.cls = _autograd_cls()
    return _Lazy.cls.apply(q, k, v)


def __getattr__(name):
    if name == "CausalAttention":
        if _Lazy.cls is None:
            _Lazy.cls = _autograd_cls()
        return _Lazy.cls
    raise AttributeError(name)
