"""torch autograd wrapper of the scan.

Mirrors the autodiff node of burn-mamba ``mamba3/quat_scan/backward.rs``
(``impl Mamba3QuatScanBackendExt for Autodiff``, ``quat_cumprod``, and the
``QuatScanBackward`` node with its ``State``): the forward runs the scan; when
gradients are tracked it keeps only the leaves ``q`` and ``init``, and the
backward recomputes from them (``quat_cumprod_bwd``).  Untracked calls keep
nothing.

``save_carries=True`` keeps the chunk carries as well (1/64 of ``q``): the
forward writes them (``quat_cumprod_fwd_carries``) and the backward starts
from them (``quat_cumprod_bwd_carries``) instead of recomputing the forward.
The page keeps only the leaves on purpose; this is the measured alternative.

``quat_cumprod_recalculated`` also returns the final carry ``cum[:, -1]`` as a
slice of ``cum``.  As in the page's module documentation, its cotangent then
reaches the node already added into ``d_cum[:, S-1]``; the node itself has a
single output.
"""
from __future__ import annotations

import torch

from . import quat_cumprod_bwd, quat_cumprod_bwd_carries, quat_cumprod_fwd, quat_cumprod_fwd_carries

__all__ = ["QuatCumprod", "quat_cumprod", "quat_cumprod_recalculated"]


class QuatCumprod(torch.autograd.Function):
    """``cum = quat_cumprod(q, init)``: forward and recompute backward in the CUDA library."""

    @staticmethod
    def forward(ctx, q, init, save_carries: bool, tracked: bool):
        # (Gradient mode is off inside forward: `tracked` is decided by the caller.)
        q = q.contiguous()
        init = init.contiguous()
        ctx.save_carries = bool(save_carries) and tracked
        if ctx.save_carries:
            cum, carries = quat_cumprod_fwd_carries(q, init)
            ctx.save_for_backward(q, carries)
        else:
            cum = quat_cumprod_fwd(q, init)
            if tracked:
                ctx.save_for_backward(q, init)
        return cum

    @staticmethod
    def backward(ctx, d_cum):
        d_cum = d_cum.contiguous()
        if ctx.save_carries:
            q, carries = ctx.saved_tensors
            d_q, d_init = quat_cumprod_bwd_carries(q, carries, d_cum)
        else:
            q, init = ctx.saved_tensors
            d_q, d_init = quat_cumprod_bwd(q, init, d_cum)
        return (d_q if ctx.needs_input_grad[0] else None,
                d_init if ctx.needs_input_grad[1] else None,
                None, None)


def quat_cumprod(q, init, *, save_carries: bool = False):
    """Differentiable scan: ``q`` [B,S,H,J,4] and ``init`` [B,H,J,4] fp32 CUDA -> ``cum``."""
    tracked = torch.is_grad_enabled() and (q.requires_grad or init.requires_grad)
    return QuatCumprod.apply(q, init, save_carries, tracked)


def quat_cumprod_recalculated(q, init, *, save_carries: bool = False):
    """``(cum, final_carry)`` with ``final_carry = cum[:, -1]`` (a slice of ``cum``)."""
    cum = quat_cumprod(q, init, save_carries=save_carries)
    return cum, cum[:, -1]
