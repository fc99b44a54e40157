"""GB300-native (sm_103a) FlashAttention forward/backward behind a C ABI.

Public Python surface (thin wrappers over include/fa.h):

    fa_fwd(q, k, v, out, lse, softmax_scale, causal, window_left, window_right, softcap)
    fa_bwd(dout, q, k, v, out, lse, dq, dk, dv, softmax_scale, causal, window_left,
           window_right, softcap, deterministic, workspace=None)
    attention_forward(q, k, v, ...)  -> (out, lse)            allocates outputs with torch
    attention_backward(dout, q, k, v, out, lse, ...) -> (dq, dk, dv)
    flash_attn_func(q, k, v, ...) / flash_attn_varlen_func(...)   torch.autograd functions

Layouts: q/out/dout/dq (B, Sq, H, D); k/v/dk/dv (B, Sk, Hk, D); all of one 16-bit type, bf16
or f16; lse (B, H, Sq) fp32 natural log.  All compute runs in libfa_gb300.so.
"""

from __future__ import annotations

import math

import torch

from ._abi import (FaError, alloc_bwd_workspace, bwd_blocksparse_workspace_size,
                   bwd_varlen_workspace_size, bwd_workspace_size, bwd_workspace_size_dv, fa_bwd, fa_bwd_blocksparse,
                   fa_bwd_status, fa_bwd_varlen, fa_fwd, fa_fwd_blocksparse, fa_fwd_varlen, load)

from .autograd import flash_attn_func, flash_attn_varlen_func

__all__ = ["FaError", "alloc_bwd_workspace", "attention_backward", "attention_backward_varlen",
           "flash_attn_func", "flash_attn_varlen_func",
           "attention_forward", "attention_forward_varlen", "bwd_varlen_workspace_size",
           "bwd_workspace_size", "bwd_workspace_size_dv", "fa_bwd", "fa_bwd_status", "fa_bwd_varlen", "fa_fwd",
           "fa_fwd_varlen", "load", "fa_fwd_blocksparse", "fa_bwd_blocksparse",
           "bwd_blocksparse_workspace_size"]


def _scale(q, softmax_scale):
    return softmax_scale if softmax_scale is not None else 1.0 / math.sqrt(q.shape[-1])


def attention_forward(q, k, v, softmax_scale=None, causal=False, window_left=-1, window_right=-1,
                      softcap=0.0):
    """out (B, Sq, H, Dv) and lse (B, H, Sq); Dv is v's head dim (it may differ from q's)."""
    B, Sq, H, D = q.shape
    out = q.new_empty(B, Sq, H, v.shape[3])
    lse = torch.empty(B, H, Sq, dtype=torch.float32, device=q.device)
    fa_fwd(q, k, v, out, lse, _scale(q, softmax_scale), causal, window_left, window_right, softcap)
    return out, lse


def attention_backward(dout, q, k, v, out, lse, softmax_scale=None, causal=False, window_left=-1,
                       window_right=-1, softcap=0.0, deterministic=False, workspace=None):
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    fa_bwd(dout, q, k, v, out, lse, dq, dk, dv, _scale(q, softmax_scale), causal, window_left,
           window_right, softcap, deterministic, workspace)
    return dq, dk, dv


def attention_forward_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                             softmax_scale=None, causal=False, window_left=-1, window_right=-1,
                             softcap=0.0, seqused_q=None, seqused_k=None):
    """Packed sequences: q (total_q, H, D), k / v (total_k, Hk, D), int32 device offsets of
    length batch + 1, optional int32 device used lengths (seqused_q / seqused_k, length
    batch).  Returns out (total_q, H, D) and lse (H, total_q); rows past a sequence's used
    length are 0 in out and +inf in lse."""
    padded = seqused_q is not None or seqused_k is not None
    out = torch.zeros_like(q) if padded else torch.empty_like(q)
    lse = (torch.full if padded else torch.empty)(
        (q.shape[1], q.shape[0]), *((float("inf"),) if padded else ()), dtype=torch.float32,
        device=q.device)
    fa_fwd_varlen(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                  _scale(q, softmax_scale), causal, window_left, window_right, softcap,
                  seqused_q=seqused_q, seqused_k=seqused_k)
    return out, lse


def attention_backward_varlen(dout, q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q,
                              max_seqlen_k, softmax_scale=None, causal=False, window_left=-1,
                              window_right=-1, softcap=0.0, deterministic=False, workspace=None,
                              seqused_q=None, seqused_k=None):
    """Packed sequences (layouts of attention_forward_varlen).  Returns dq, dk, dv; rows
    past a sequence's used length are 0."""
    dq = torch.zeros_like(q) if seqused_q is not None else torch.empty_like(q)
    dk = torch.zeros_like(k)
    dv = torch.zeros_like(v)
    fa_bwd_varlen(dout, q, k, v, out, lse, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, max_seqlen_q,
                  max_seqlen_k, _scale(q, softmax_scale), causal, window_left, window_right,
                  softcap, deterministic, workspace, seqused_q=seqused_q, seqused_k=seqused_k)
    return dq, dk, dv
