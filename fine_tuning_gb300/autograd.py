"""Optional autograd wrappers around the ftk ops, and the LoRA+ learning-rate
rule for building optimizer parameter groups.

Each Function runs the library's forward kernel, saves what the backward
kernel needs, and calls the backward kernel: argument marshalling only, no
arithmetic of its own (weight gradients, which the kernels produce in fp32,
are cast to the weight's dtype as autograd requires).

LoRA+ ("Chronicals", arXiv 2601.02609, abstract, optimisation (3)): the
adapter matrix B of every LoRA pair learns at 16 times the rate of A.
``lora_plus_param_groups`` turns that rule into parameter groups for any
torch optimizer.
"""
from __future__ import annotations

from typing import Iterable, List, Optional, Tuple

import torch

from . import ftk

LORA_PLUS_RATIO = 16.0


class RMSNorm(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, w, eps: float):
        y, rstd = ftk.rmsnorm_fwd(x, w, eps)
        ctx.save_for_backward(x, w, rstd)
        ctx.eps = eps
        return y

    @staticmethod
    def backward(ctx, dy):
        x, w, rstd = ctx.saved_tensors
        dx, dw = ftk.rmsnorm_bwd(dy.contiguous(), x, w, rstd, ctx.eps)
        return dx, dw.to(w.dtype), None


class AddRMSNorm(torch.autograd.Function):
    """(h, y) = (x + res, rmsnorm(x + res) * w)."""

    @staticmethod
    def forward(ctx, x, res, w, eps: float):
        h, y, rstd = ftk.rmsnorm_add_fwd(x, res, w, eps)
        ctx.save_for_backward(h, w, rstd)
        ctx.eps = eps
        return h, y

    @staticmethod
    def backward(ctx, dh, dy):
        h, w, rstd = ctx.saved_tensors
        dh = torch.zeros_like(h) if dh is None else dh.contiguous()
        dy = torch.zeros_like(h) if dy is None else dy.contiguous()
        dx, dw = ftk.rmsnorm_add_bwd(dy, dh, h, w, rstd, ctx.eps)
        return dx, dx, dw.to(w.dtype), None


class SwiGLU(torch.autograd.Function):
    @staticmethod
    def forward(ctx, g, u):
        ctx.save_for_backward(g, u)
        return ftk.swiglu_fwd(g, u)

    @staticmethod
    def backward(ctx, dh):
        g, u = ctx.saved_tensors
        dg, du = ftk.swiglu_bwd(dh.contiguous(), g, u)
        return dg, du


class QKRope(torch.autograd.Function):
    """Rotates copies of q [T, Hq, D] and k [T, Hkv, D]; inv_freq (host, D/2)
    replaces theta when given."""

    @staticmethod
    def forward(ctx, q, k, cu_seqlens, theta: float, inv_freq=None):
        q, k = q.clone(), k.clone()
        if inv_freq is None:
            ftk.qk_rope_fwd(q, k, cu_seqlens, theta)
        else:
            ftk.qk_rope_freq_fwd(q, k, cu_seqlens, inv_freq)
        ctx.save_for_backward(cu_seqlens)
        ctx.theta, ctx.inv_freq = theta, inv_freq
        return q, k

    @staticmethod
    def backward(ctx, dq, dk):
        (cu,) = ctx.saved_tensors
        dq, dk = dq.contiguous().clone(), dk.contiguous().clone()
        if ctx.inv_freq is None:
            ftk.qk_rope_bwd(dq, dk, cu, ctx.theta)
        else:
            ftk.qk_rope_freq_bwd(dq, dk, cu, ctx.inv_freq)
        return dq, dk, None, None, None


class QKNormRope(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, wq, wk, cu_seqlens, eps: float, theta: float, inv_freq=None):
        qo, ko, rq, rk = ftk.qk_norm_rope_fwd(q, k, wq, wk, cu_seqlens, eps, theta=theta,
                                              inv_freq=inv_freq)
        ctx.save_for_backward(q, k, wq, wk, rq, rk, cu_seqlens)
        ctx.eps, ctx.theta, ctx.inv_freq = eps, theta, inv_freq
        return qo, ko

    @staticmethod
    def backward(ctx, dq, dk):
        q, k, wq, wk, rq, rk, cu = ctx.saved_tensors
        gq, gk, dwq, dwk = ftk.qk_norm_rope_bwd(dq.contiguous(), dk.contiguous(), q, k, wq, wk,
                                                rq, rk, cu, ctx.eps, theta=ctx.theta,
                                                inv_freq=ctx.inv_freq)
        return gq, gk, dwq.to(wq.dtype), dwk.to(wk.dtype), None, None, None, None


class CrossEntropyHead(torch.autograd.Function):
    """Mean cross-entropy of the logits h W^T against y (int32; y outside
    [0, V) is ignored), the logits never materialised."""

    @staticmethod
    def forward(ctx, h, W, y):
        loss, lse = ftk.cce_fwd(h, W, y)
        ctx.save_for_backward(h, W, y, lse)
        return loss.reshape(())

    @staticmethod
    def backward(ctx, dloss):
        h, W, y, lse = ctx.saved_tensors
        g = dloss.reshape(1).to(torch.float32).contiguous()
        dh, dW = ftk.cce_bwd(h, W, y, lse, g)
        return dh, dW.to(W.dtype), None


def rmsnorm(x, w, eps: float):
    return RMSNorm.apply(x, w, eps)


def add_rmsnorm(x, res, w, eps: float):
    return AddRMSNorm.apply(x, res, w, eps)


def swiglu(g, u):
    return SwiGLU.apply(g, u)


def qk_rope(q, k, cu_seqlens, theta: float, inv_freq=None):
    return QKRope.apply(q, k, cu_seqlens, theta, inv_freq)


def qk_norm_rope(q, k, wq, wk, cu_seqlens, eps: float, theta: float, inv_freq=None):
    return QKNormRope.apply(q, k, wq, wk, cu_seqlens, eps, theta, inv_freq)


def cross_entropy_head(h, W, y):
    return CrossEntropyHead.apply(h, W, y)


def _is_lora_b(name: str) -> bool:
    parts = name.replace("/", ".").split(".")
    return any(p in ("lora_B", "lora_b", "B") for p in parts[-3:]) or name.endswith("lora_B")


def lora_plus_param_groups(named_parameters: Iterable[Tuple[str, torch.nn.Parameter]],
                           lr: float, ratio: float = LORA_PLUS_RATIO,
                           weight_decay: Optional[float] = None) -> List[dict]:
    """Parameter groups for the LoRA+ rule: every LoRA B matrix (a parameter
    whose dotted name has a ``lora_B`` (or ``B``) component) at lr * ratio,
    everything else trainable (the A matrices, biases, ...) at lr.  Frozen
    parameters are left out.  Pass the result to any torch optimizer."""
    a_params, b_params = [], []
    for name, p in named_parameters:
        if not p.requires_grad:
            continue
        (b_params if _is_lora_b(name) else a_params).append(p)
    groups = []
    extra = {} if weight_decay is None else {"weight_decay": weight_decay}
    if a_params:
        groups.append({"params": a_params, "lr": lr, **extra})
    if b_params:
        groups.append({"params": b_params, "lr": lr * ratio, **extra})
    return groups
