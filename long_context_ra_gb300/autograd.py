"""Differentiable ring attention for PyTorch training.

`attention` (one device, the virtual ring) and `ring_attention` (one rank
per device, the ring of `long_context_ra_gb300.ring`) are torch.autograd
Functions: the forward is the library's forward and the backward its
backward ("Ring attention, explained", step 6: the backward runs on the same
ring).  They hold no arithmetic of their own; out is differentiable, lse is
returned as a non-differentiable tensor (the backward takes the gradient of
out only)."""
from __future__ import annotations

import torch

from . import ra_backward, ra_forward, ra_forward_causal


class _Attention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, P, layout):
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        if layout is None:
            out, lse = ra_forward(q, k, v, P)
        else:
            out, lse = ra_forward_causal(q, k, v, P, layout=layout)
        ctx.save_for_backward(q, k, v, out, lse)
        ctx.P, ctx.layout = P, layout
        ctx.mark_non_differentiable(lse)
        return out, lse

    @staticmethod
    def backward(ctx, dout, _dlse):
        q, k, v, out, lse = ctx.saved_tensors
        dq, dk, dv = ra_backward(q, k, v, out, dout.contiguous(), lse, ctx.P, causal=ctx.layout)
        return dq, dk, dv, None, None


def attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, P: int = 1,
              causal: str | None = None):
    """Differentiable attention over [B, H, N, d] tensors on one device, in
    ring order over P blocks (any P dividing N gives the same result).
    causal: None, or the layout of the causal ring ("contiguous", "zigzag",
    "striped").  Returns (out, lse); gradients flow through out."""
    return _Attention.apply(q, k, v, P, causal)


class _RingAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, group, causal, layout, ops, bops):
        from .ring import ring_forward

        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        out, lse = ring_forward(q, k, v, group=group, ops=ops, causal=causal, layout=layout)
        ctx.save_for_backward(q, k, v, out, lse)
        ctx.args = (group, causal, layout, bops)
        ctx.mark_non_differentiable(lse)
        return out, lse

    @staticmethod
    def backward(ctx, dout, _dlse):
        from .ring import ring_backward

        q, k, v, out, lse = ctx.saved_tensors
        group, causal, layout, bops = ctx.args
        dq, dk, dv = ring_backward(q, k, v, out, dout.contiguous(), lse, group=group, ops=bops,
                                   causal=causal, layout=layout)
        return dq, dk, dv, None, None, None, None, None


def ring_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, group=None,
                   causal: bool = False, layout: str = "contiguous", ops=None, bops=None):
    """Differentiable attention of this rank's block over the whole sequence
    held by the ranks of `group` (see `ring.ring_forward`): the forward ring
    passes K/V blocks, and the backward ring passes them with their dK, dV
    accumulators.  Every rank calls it with blocks of the same shape, and
    every rank's backward runs when any rank's does (the ring's sends pair
    up).  `ops` / `bops` replace the forward / backward operations (default:
    the library's kernels).  Returns (out, lse) of the block."""
    return _RingAttention.apply(q, k, v, group, causal, layout, ops, bops)
