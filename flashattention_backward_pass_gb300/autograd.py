"""torch.autograd entry points over the C ABI: `flash_attn_func` and
`flash_attn_varlen_func` (the call-trace page's `flash_attn_func` -> `_flash_attn_forward`
/ `_flash_attn_backward` pair, and the Triton page's `flash_attn_varlen_func`).

The forward saves q, k, v, out and the natural-log LSE; the backward calls fa_bwd /
fa_bwd_varlen with them (dQ, dK, dV written by the library's kernels).  Every step runs
in libfa_gb300.so: these classes only allocate outputs and pass tensors through.

A bounded device-side wait that runs out (FA_ERR_DEVICE_TIMEOUT) is recorded in the
backward's workspace, not returned by the launch.  With the environment variable
FA_CHECK_DEVICE_STATUS=1 the backward reads that status word after each call (a stream
synchronisation) and raises FaError when it is non-zero; by default it does not check,
so a timed-out call would leave incomplete gradients without an error.
"""

from __future__ import annotations

import math
import os

import torch

from . import _abi


def _check_status(workspace):
    if os.environ.get("FA_CHECK_DEVICE_STATUS", "0") not in ("", "0"):
        st = _abi.fa_bwd_status(workspace)
        if st != 0:
            raise _abi.FaError(-11, f"backward device status {st}")


def _scale(q, softmax_scale):
    return softmax_scale if softmax_scale is not None else 1.0 / math.sqrt(q.shape[-1])


class FlashAttnFunc(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, softmax_scale, causal, window_left, window_right, softcap,
                deterministic):
        q, k, v = (t if t.stride(-1) == 1 else t.contiguous() for t in (q, k, v))
        B, Sq, H, _ = q.shape
        out = q.new_empty(B, Sq, H, v.shape[3])
        lse = torch.empty(B, H, Sq, dtype=torch.float32, device=q.device)
        _abi.fa_fwd(q, k, v, out, lse, softmax_scale, causal, window_left, window_right, softcap)
        ctx.save_for_backward(q, k, v, out, lse)
        ctx.args = (softmax_scale, causal, window_left, window_right, softcap, deterministic)
        return out

    @staticmethod
    def backward(ctx, dout):
        q, k, v, out, lse = ctx.saved_tensors
        scale, causal, wl, wr, softcap, det = ctx.args
        dout = dout if dout.stride(-1) == 1 else dout.contiguous()
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = _abi.fa_bwd(dout, q, k, v, out, lse, dq, dk, dv, scale, causal, wl, wr, softcap, det)
        _check_status(ws)
        return dq, dk, dv, None, None, None, None, None, None


def flash_attn_func(q, k, v, softmax_scale=None, causal=False, window_left=-1, window_right=-1,
                    softcap=0.0, deterministic=False):
    """Attention with gradients: q (B, Sq, H, D), k / v (B, Sk, Hk, D), bf16 or f16.
    Returns out (B, Sq, H, D); its backward produces dq, dk, dv through fa_bwd."""
    return FlashAttnFunc.apply(q, k, v, _scale(q, softmax_scale), bool(causal), int(window_left),
                               int(window_right), float(softcap), bool(deterministic))


class FlashAttnVarlenFunc(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                softmax_scale, causal, window_left, window_right, softcap, deterministic,
                seqused_q, seqused_k):
        q, k, v = (t if t.stride(-1) == 1 else t.contiguous() for t in (q, k, v))
        padded = seqused_q is not None or seqused_k is not None
        out = torch.zeros_like(q) if padded else torch.empty_like(q)
        lse = torch.empty(q.shape[1], q.shape[0], dtype=torch.float32, device=q.device)
        _abi.fa_fwd_varlen(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q,
                           max_seqlen_k, softmax_scale, causal, window_left, window_right,
                           softcap, seqused_q=seqused_q, seqused_k=seqused_k)
        ctx.save_for_backward(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k)
        ctx.used = (seqused_q, seqused_k)
        ctx.args = (max_seqlen_q, max_seqlen_k, softmax_scale, causal, window_left,
                    window_right, softcap, deterministic)
        return out

    @staticmethod
    def backward(ctx, dout):
        q, k, v, out, lse, cu_q, cu_k = ctx.saved_tensors
        mq, mk, scale, causal, wl, wr, softcap, det = ctx.args
        dout = dout if dout.stride(-1) == 1 else dout.contiguous()
        uq, uk = ctx.used
        dq = torch.zeros_like(q) if uq is not None else torch.empty_like(q)
        dk, dv = torch.zeros_like(k), torch.zeros_like(v)
        ws = _abi.fa_bwd_varlen(dout, q, k, v, out, lse, dq, dk, dv, cu_q, cu_k, mq, mk, scale,
                                causal, wl, wr, softcap, det, seqused_q=uq, seqused_k=uk)
        _check_status(ws)
        return (dq, dk, dv) + (None,) * 12


def flash_attn_varlen_func(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                           softmax_scale=None, causal=False, window_left=-1, window_right=-1,
                           softcap=0.0, deterministic=False, seqused_q=None, seqused_k=None):
    """Packed sequences with gradients: q (total_q, H, D), k / v (total_k, Hk, D), int32
    device offsets of length batch + 1, optional int32 device used lengths of length batch
    (rows past them are padding: out and the gradients are 0 there).  Returns out
    (total_q, H, D)."""
    return FlashAttnVarlenFunc.apply(q, k, v, cu_seqlens_q, cu_seqlens_k, int(max_seqlen_q),
                                     int(max_seqlen_k), _scale(q, softmax_scale), bool(causal),
                                     int(window_left), int(window_right), float(softcap),
                                     bool(deterministic), seqused_q, seqused_k)
