"""Autograd wrapper: the fused call as a differentiable loss.

The LM head is the last layer, so its gradients can be produced during the
forward pass. The FLCE page ("Fused Linear Cross-Entropy: LLM 학습 logits
메모리 병목 없애기", section "FLCE의 핵심 아이디어") quotes Liger's source
comment to that effect. The forward here runs the whole fused forward +
backward in the library and keeps dx and dW. The backward only scales them by
the incoming gradient of the (scalar) loss, which is 1 in the usual
`loss.backward()`, and then no arithmetic runs at all. The pattern is the
hand-written forward/backward pair the Unsloth page shows for its fused
kernels ("Unsloth 심층 아키텍처 …", section "소스코드 레벨 아키텍처 구현 패턴").
"""
from __future__ import annotations

import torch

from .flce import FLCE

_handles = {}


def _handle(device: torch.device, dtype: torch.dtype, dlogits_mode: str = "auto",
            hbm_budget_bytes: int = 0) -> FLCE:
    key = (device.index or 0, dtype, dlogits_mode, hbm_budget_bytes)
    if key not in _handles:
        _handles[key] = FLCE("bf16" if dtype == torch.bfloat16 else "fp32", key[0],
                             hbm_budget_bytes=hbm_budget_bytes, dlogits_mode=dlogits_mode)
    return _handles[key]


class LinearCrossEntropyFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, W, t, ignore_index: int, chunk: int, reduction: str, handle,
                sync_free: bool = False, dlogits_mode: str = "auto", hbm_budget_bytes: int = 0):
        h = handle if handle is not None else _handle(x.device, x.dtype, dlogits_mode, hbm_budget_bytes)
        if reduction not in ("mean", "sum"):
            raise ValueError("reduction must be 'mean' or 'sum'")
        ctx.sync_free = sync_free
        if sync_free:
            # no host synchronisation anywhere: the loss stays on the device
            # (NaN after a device-side error) and the gradients are always
            # scaled by the incoming gradient on the device
            loss, n_valid, dx, dW = h.forward_backward_async(
                x.contiguous(), W.contiguous(), t.contiguous(), ignore_index=ignore_index,
                chunk=chunk)
            scale = n_valid.float() if reduction == "sum" else torch.ones((), device=x.device)
            ctx.save_for_backward(dx, dW, scale)
            return loss * scale
        loss, dx, dW = h.forward_backward(x.contiguous(), W.contiguous(), t.contiguous(),
                                          ignore_index=ignore_index, chunk=chunk)
        scale = 1.0
        if reduction == "sum":
            # the library returns the mean over the n_valid counted tokens
            scale = float((t != ignore_index).sum().item())
        ctx.scale = scale
        ctx.save_for_backward(dx, dW)
        return torch.tensor(loss * scale, dtype=torch.float32, device=x.device)

    @staticmethod
    def backward(ctx, grad_out):
        if ctx.sync_free:
            dx, dW, scale = ctx.saved_tensors
            g = grad_out * scale
            gx = dx * g.to(dx.dtype) if ctx.needs_input_grad[0] else None
            gW = dW * g if ctx.needs_input_grad[1] else None
            return gx, gW, None, None, None, None, None, None, None, None
        dx, dW = ctx.saved_tensors
        g = grad_out * ctx.scale
        if ctx.needs_input_grad[0]:
            gx = dx if (ctx.scale == 1.0 and bool(grad_out == 1)) else dx * g.to(dx.dtype)
        else:
            gx = None
        if ctx.needs_input_grad[1]:
            gW = dW if (ctx.scale == 1.0 and bool(grad_out == 1)) else dW * g
        else:
            gW = None
        return gx, gW, None, None, None, None, None, None, None, None


def linear_cross_entropy(x: torch.Tensor, W: torch.Tensor, t: torch.Tensor,
                         ignore_index: int = -100, reduction: str = "mean", chunk: int = 0,
                         handle: FLCE = None, sync_free: bool = False, dlogits_mode: str = "auto",
                         hbm_budget_bytes: int = 0) -> torch.Tensor:
    """Cross-entropy of x·Wᵀ against t, fused: the N x V logits never exist.

    x: (N, H) bf16 or fp32 on a GB300; W: (V, H) same dtype; t: (N,) int64.
    Returns a 0-dim fp32 tensor. `loss.backward()` gives x.grad and W.grad;
    W.grad is computed in fp32 and cast by autograd to W's dtype.

    sync_free=True never blocks the host (a step can then be captured in a
    CUDA graph): the loss is NaN after a device-side error, which
    FLCE.async_status() reports, and the backward always scales dx and dW by
    the incoming gradient (one extra pass over dW). The default synchronises
    once per call, raises on errors at once, and skips that pass when the
    incoming gradient is 1.

    Without a `handle`, one is kept per (device, dtype, dlogits_mode,
    hbm_budget_bytes): dlogits_mode "slabs" with a small budget gives the
    vocabulary-slab backward, whose workspace does not grow with V.
    """
    return LinearCrossEntropyFunction.apply(x, W, t, ignore_index, chunk, reduction, handle,
                                            sync_free, dlogits_mode, hbm_budget_bytes)
