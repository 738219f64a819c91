"""PyTorch autograd wrappers: the library's forward and backward entry points
as one differentiable function (argument marshalling only; both directions
run in the library's kernels).

    o = linear_attention(q, k, v, causal=True)     # q, k: [B,H,N,Dk], v: [B,H,N,Dv]
    o.backward(g)                                   # la_causal_bwd fills q.grad, k.grad, v.grad

The backward takes Dk, Dv <= 64 (the library refuses wider heads with
LA_ERR_UNSUPPORTED). Gradients have the inputs' dtype.
"""
import torch

from . import (LA_PHI_ELU1, la_causal_bwd, la_causal_fwd, la_noncausal_bwd,
               la_noncausal_fwd)


class _LinearAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, causal, eps, phi):
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        fwd = la_causal_fwd if causal else la_noncausal_fwd
        o = fwd(q, k, v, eps=eps, phi=phi)
        ctx.save_for_backward(q, k, v)
        ctx.causal, ctx.eps, ctx.phi = causal, eps, phi
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v = ctx.saved_tensors
        bwd = la_causal_bwd if ctx.causal else la_noncausal_bwd
        dq, dk, dv = bwd(q, k, v, do.contiguous().to(v.dtype), eps=ctx.eps, phi=ctx.phi)
        return dq, dk, dv, None, None, None


def linear_attention(q, k, v, causal=True, eps=1e-6, phi=LA_PHI_ELU1):
    """Differentiable elu+1 linear attention (or another feature map via `phi`)."""
    return _LinearAttention.apply(q, k, v, bool(causal), float(eps), int(phi))
