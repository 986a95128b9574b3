"""linear_logp as an autograd operation (deterministic_token_logprob_gb300.linear_logp): its
forward and the gradients autograd hands to h and W are the bits of the direct C-ABI calls
(rlk_linear_logp_fwd, then rlk_linear_logp_bwd with g = dL/dlogp)."""
import numpy as np
import pytest
import torch

import workloads
from gpu_util import dev, dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rlk():
    from deterministic_token_logprob_gb300 import build
    build.build()
    import deterministic_token_logprob_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def test_autograd_gradients_are_the_direct_calls_bits(rlk):
    T, H, V, Vt = 300, 512, 20480, 20000
    d = workloads.make_inputs(workloads.Workload("ag", T=T, H=H, V=V, V_true=Vt, seed=61))
    h = dev_bf16(d["h"]).requires_grad_()
    W = dev_bf16(d["W"]).requires_grad_()
    y = dev(d["y"])
    adv = torch.from_numpy(np.random.default_rng(62).standard_normal(T).astype(np.float32)).cuda()
    logp = rlk.linear_logp(h, W, y, Vt)
    loss = -(adv * logp).sum() / T            # a policy-gradient-style loss on top of logp
    loss.backward()
    ref_logp, ref_lse = rlk.linear_logp_fwd(h.detach(), W.detach(), y, Vt)
    g = (-adv / T).contiguous()               # dL/dlogp of that loss
    ref_dH, ref_dW = rlk.linear_logp_bwd(h.detach(), W.detach(), y, ref_lse, g, Vt)
    torch.cuda.synchronize()
    assert logp.dtype == torch.float32 and torch.equal(logp.detach(), ref_logp)
    assert h.grad.dtype == torch.bfloat16 and torch.equal(h.grad, ref_dH)
    assert W.grad.dtype == torch.bfloat16 and torch.equal(W.grad, ref_dW.to(torch.bfloat16))


def test_autograd_only_computes_the_gradients_asked_for(rlk):
    T, H, V = 64, 256, 4096
    d = workloads.make_inputs(workloads.TINY)
    h = dev_bf16(d["h"]).requires_grad_()
    W = dev_bf16(d["W"])                       # frozen LM head: no dW
    y = dev(d["y"])
    logp = rlk.linear_logp(h, W, y)            # V_true defaults to V
    logp.sum().backward()
    _, lse = rlk.linear_logp_fwd(h.detach(), W, y, V)
    ref_dH, _ = rlk.linear_logp_bwd(h.detach(), W, y, lse, torch.ones(T, device="cuda"), V,
                                    want_dW=False)
    torch.cuda.synchronize()
    assert W.grad is None and torch.equal(h.grad, ref_dH)
