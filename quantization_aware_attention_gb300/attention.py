"""Torch-facing API over the C ABI: output allocation, the backward workspace and the
autograd Function.  torch supplies device memory and streams only; every step of the
computation runs in the library's CUDA kernels.

``attention(q, k, v, causal, sm_scale, quant_mode)`` returns the quantized output O_q
and, under autograd, back-propagates through the straight-through estimator: the
saved O_hp and log-sum-exp let the backward rematerialize P ("support for pytorch
autograd": rematerialization as in FlashAttention; "attn_qat_train.py",
_attention.forward saves q, k, v, O and M).
"""

from __future__ import annotations

import math
import os

import torch

from . import capi


def _check(t: torch.Tensor, name: str, shape=None, dtype=torch.bfloat16) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (this library has no CPU path)")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _dims(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor):
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, H, N, D]")
    B, H, Nq, D = q.shape
    Nkv = k.shape[2]
    _check(q, "q")
    _check(k, "k", (B, H, Nkv, D))
    _check(v, "v", (B, H, Nkv, D))
    return B, H, Nq, Nkv, D


def _raise(st: capi.Status, what: str) -> None:
    if st != capi.Status.OK:
        raise capi.QatError(st, what)


def _check_enabled(check: bool | None) -> bool:
    """Whether to read the device error word after each call: the argument, else the
    environment variable QAT_CHECK_STATUS=1."""
    if check is not None:
        return bool(check)
    return os.environ.get("QAT_CHECK_STATUS", "0") == "1"


def check_device_status(what: str = "QAT attention") -> None:
    """Synchronizes the current stream and raises QatError if a kernel's bounded wait
    expired since the last check (the kernel then returned early and its outputs are
    incomplete).  The read clears the error word."""
    _raise(capi.qat_attn_device_status(), what)


def qat_attention_forward(q, k, v, causal: bool = False, sm_scale: float | None = None,
                          quant_mode: int = capi.QUANT_P_FP8E4M3_ROW_TILE64):
    """Returns (o_q, o_hp, lse): bf16 [B,H,Nq,D], bf16 [B,H,Nq,D], fp32 [B,H,Nq] (base 2)."""
    B, H, Nq, Nkv, D = _dims(q, k, v)
    sm_scale = 1.0 / math.sqrt(D) if sm_scale is None else float(sm_scale)
    o_q = torch.empty_like(q)
    o_hp = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        st = capi.qat_attn_fwd(q, k, v, o_q, o_hp, lse, B, H, Nq, Nkv, D, sm_scale,
                               int(causal), quant_mode)
    _raise(st, "qat_attn_fwd")
    return o_q, o_hp, lse


def qat_attention_backward(q, k, v, o_hp, lse, do, causal: bool = False,
                           sm_scale: float | None = None,
                           quant_mode: int = capi.QUANT_P_FP8E4M3_ROW_TILE64,
                           workspace: torch.Tensor | None = None,
                           k_mean: torch.Tensor | None = None):
    """Returns (dq, dk, dv) of L = <dO, O_hp> (straight-through estimator; quant_mode 2:
    the page's backward, with the forward's O_q passed as ``o_hp``).  With ``k_mean``
    (fp32 [D], smooth_k's channel mean; k is the smoothed key) dQ gets the page's
    SMOOTH_K term."""
    B, H, Nq, Nkv, D = _dims(q, k, v)
    _check(o_hp, "o_hp", (B, H, Nq, D))
    _check(do, "do", (B, H, Nq, D))
    _check(lse, "lse", (B, H, Nq), torch.float32)
    if k_mean is not None:
        _check(k_mean, "k_mean", (D,), torch.float32)
    sm_scale = 1.0 / math.sqrt(D) if sm_scale is None else float(sm_scale)
    ws_bytes = capi.qat_attn_bwd_workspace_bytes(B, H, Nq, Nkv, D)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    with torch.cuda.device(q.device):
        if k_mean is None:
            st = capi.qat_attn_bwd(q, k, v, o_hp, lse, do, dq, dk, dv, B, H, Nq, Nkv, D,
                                   sm_scale, int(causal), quant_mode, workspace,
                                   workspace.numel())
        else:
            st = capi.qat_attn_bwd_smooth_k(q, k, v, o_hp, lse, do, dq, dk, dv, k_mean, B, H, Nq,
                                            Nkv, D, sm_scale, int(causal), quant_mode,
                                            workspace, workspace.numel())
    _raise(st, "qat_attn_bwd")
    return dq, dk, dv


def qat_subtract_mean(x: torch.Tensor, mean: torch.Tensor) -> torch.Tensor:
    """bf16(x - mean) per channel: smooth_k's subtraction without the quantization."""
    B, H, N, D = x.shape
    _check(x, "x")
    _check(mean, "mean", (D,), torch.float32)
    out = torch.empty_like(x)
    with torch.cuda.device(x.device):
        _raise(capi.qat_subtract_mean(x, mean, out, B, H, N, D), "qat_subtract_mean")
    return out


def qat_prepare_qkv(q, k, v, smooth_k: bool = True):
    """The page's IS_QAT inputs: fake-quantized copies of q, k, v (FP8 E4M3, one absmax
    scale per (head, 32-token block)); with smooth_k the per-channel mean of K over
    batch, heads and tokens is subtracted before K is quantized ("attn_qat_train.py",
    _attention.forward).  Returns (q_fq, k_fq, v_fq, k_mean or None)."""
    B, H, Nq, Nkv, D = _dims(q, k, v)
    k_mean = None
    with torch.cuda.device(q.device):
        if smooth_k:
            k_mean = torch.empty(D, dtype=torch.float32, device=q.device)
            _raise(capi.qat_channel_mean(k, k_mean, B, H, Nkv, D), "qat_channel_mean")
        out = []
        for x, n, m in ((q, Nq, None), (k, Nkv, k_mean), (v, Nkv, None)):
            y = torch.empty_like(x)
            _raise(capi.qat_fake_quant_tokens(x, m, y, None, B, H, n, D), "qat_fake_quant_tokens")
            out.append(y)
    return out[0], out[1], out[2], k_mean


class QATAttention(torch.autograd.Function):
    """Forward returns O_q; backward returns dq, dk, dv through the straight-through
    estimator (gradients of O_hp), or the page's backward with quant_mode 2."""

    @staticmethod
    def forward(ctx, q, k, v, causal=False, sm_scale=None,
                quant_mode=capi.QUANT_P_FP8E4M3_ROW_TILE64, qkv_quant=False, smooth_k=False,
                use_qat_qkv_backward=True, check=None):
        k_mean = None
        q_bwd, k_bwd, v_bwd = q, k, v
        if qkv_quant:  # attention runs on fake-quantized inputs; gradients pass straight
            qf, kf, vf, k_mean = qat_prepare_qkv(q, k, v, smooth_k)
            if use_qat_qkv_backward:
                q_bwd, k_bwd, v_bwd = qf, kf, vf
            elif k_mean is not None:  # the page keeps q, k - k_mean, v for its backward
                k_bwd = qat_subtract_mean(k, k_mean)
            q, k, v = qf, kf, vf
        elif smooth_k:
            raise ValueError("smooth_k changes the result only together with qkv_quant")
        elif not use_qat_qkv_backward:
            raise ValueError("use_qat_qkv_backward=False applies only together with qkv_quant")
        ctx.check = _check_enabled(check)
        o_q, o_hp, lse = qat_attention_forward(q, k, v, causal, sm_scale, quant_mode)
        if ctx.check:
            check_device_status("qat_attn_fwd")
        # the page's backward variant forms Delta from O_q, the straight-through one from O_hp
        o_bwd = o_q if quant_mode == capi.QUANT_P_FP8E4M3_ROW_TILE64_PAGE_BWD else o_hp
        saved = (q_bwd, k_bwd, v_bwd, o_bwd, lse) + ((k_mean,) if k_mean is not None else ())
        ctx.save_for_backward(*saved)
        ctx.causal, ctx.sm_scale, ctx.quant_mode = causal, sm_scale, quant_mode
        return o_q

    @staticmethod
    def backward(ctx, do):
        q, k, v, o_bwd, lse, *rest = ctx.saved_tensors
        k_mean = rest[0] if rest else None
        dq, dk, dv = qat_attention_backward(q, k, v, o_bwd, lse, do.contiguous(), ctx.causal,
                                            ctx.sm_scale, ctx.quant_mode, k_mean=k_mean)
        if ctx.check:
            check_device_status("qat_attn_bwd")
        return dq, dk, dv, None, None, None, None, None, None, None


def attention(q, k, v, causal: bool = False, sm_scale: float | None = None,
              quant_mode: int = capi.QUANT_P_FP8E4M3_ROW_TILE64, qkv_quant: bool = False,
              smooth_k: bool = False, use_qat_qkv_backward: bool = True,
              check: bool | None = None):
    """QAT attention: the quantized output O_q, differentiable (straight-through; the
    page's own backward with quant_mode 2).

    qkv_quant additionally fake-quantizes q, k, v per 32-token block first (the page's
    full IS_QAT path), smooth_k subtracting K's channel mean before K is quantized (and
    adding the SMOOTH_K term to dQ).  With use_qat_qkv_backward=False the backward runs on
    the unquantized q, k - k_mean and v, as the page's option of that name does.
    check=True (or QAT_CHECK_STATUS=1 in the environment) synchronizes after the forward
    and the backward and raises QatError if a kernel's bounded wait expired, so that a
    call cut short is never consumed silently."""
    return QATAttention.apply(q, k, v, causal, sm_scale, quant_mode, qkv_quant, smooth_k,
                              use_qat_qkv_backward, check)
