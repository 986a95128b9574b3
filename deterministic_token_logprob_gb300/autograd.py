"""linear_logp as a PyTorch autograd operation.

``linear_logp(h, W, y, V_true)`` returns logp[t] = h[t].W[y[t]] - logsumexp_{v < V_true}(h[t].W)
(fp32 [T]) like rlk_linear_logp_fwd, and its backward, for an upstream gradient g = dL/dlogp,
calls rlk_linear_logp_bwd (the logits recomputed tile by tile, dz = g (onehot - softmax), then
dH = dz W and dW = dz^T h): the operator boundary "hidden + lm_head_weight + target_ids ->
selected logprob" with its full gradient ("Announcing RL-Kernel for vime", sections "Why the
Fused Path Wins" and "Key Capabilities"). Both directions run the library's kernels through
the C ABI; this module only saves the forward's lse for the backward and hands the gradients
to autograd. dH comes back in h's dtype (bf16, one rounding of the fp32 accumulator); dW is
computed in fp32 and autograd casts it to W's dtype for W.grad.
"""
from __future__ import annotations

import torch

from . import _binding


class LinearLogp(torch.autograd.Function):
    @staticmethod
    def forward(ctx, h, W, y, V_true: int):
        logp, lse = _binding.linear_logp_fwd(h, W, y, V_true)
        ctx.save_for_backward(h, W, y, lse)
        ctx.V_true = V_true
        return logp

    @staticmethod
    def backward(ctx, grad_logp):
        h, W, y, lse = ctx.saved_tensors
        want_dH, want_dW = ctx.needs_input_grad[0], ctx.needs_input_grad[1]
        if not (want_dH or want_dW):
            return None, None, None, None
        g = grad_logp.contiguous().to(torch.float32)
        dH, dW = _binding.linear_logp_bwd(h, W, y, lse, g, ctx.V_true, want_dH=want_dH,
                                          want_dW=want_dW)
        return dH, dW, None, None


def linear_logp(h: torch.Tensor, W: torch.Tensor, y: torch.Tensor, V_true: int = None) -> torch.Tensor:
    """Selected-token log-probabilities with autograd: bf16 h [T, H], bf16 W [V, H], int64 y [T]
    (targets in [0, V_true)); V_true defaults to V. Returns fp32 logp [T]."""
    return LinearLogp.apply(h, W, y, W.shape[0] if V_true is None else int(V_true))
