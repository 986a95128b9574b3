"""The size limits of the C ABI (RLK_MAX_VOCAB = 2^24 vocab rows, RLK_MAX_HIDDEN =
2^16 hidden units), against the oracle, and one step past each limit rejected."""
import numpy as np
import pytest
import torch

import workloads
from gpu_util import assert_grad_close, assert_logp_close, dev, dev_bf16, host_bf16_to_f64

pytestmark = pytest.mark.gpu

MAX_VOCAB = 1 << 24
MAX_HIDDEN = 1 << 16


@pytest.fixture(scope="module")
def rlk():
    from deterministic_token_logprob_gb300 import build
    build.build()
    import deterministic_token_logprob_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def test_largest_vocabulary(rlk, oracle_mod):
    # 16384 leaves -> 8 super-shards of 2048 leaves, 2048 slots each: the deepest tree
    T, H, V = 5, 64, MAX_VOCAB
    Vt = V - 77
    d = workloads.make_inputs(workloads.Workload("maxv", T=T, H=H, V=V, V_true=Vt, seed=3))
    y = d["y"].copy()
    y[0], y[1] = 0, Vt - 1                       # first and last valid columns
    h, W, yd, g = dev_bf16(d["h"]), dev_bf16(d["W"]), dev(y), dev(d["g"])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    logp, lse = rlk.linear_logp_fwd(h, W, yd, Vt, err_flag=err)
    dH, dW = rlk.linear_logp_bwd(h, W, yd, lse, g, Vt, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref_logp, ref_lse = oracle_mod.forward(d["h"], d["W"], y, Vt)
    assert_logp_close(logp.cpu().numpy(), ref_logp)
    assert_logp_close(lse.cpu().numpy(), ref_lse)
    g64 = d["g"].astype(np.float64)
    ref_dH = oracle_mod.backward_dh(d["h"], d["W"], y, g64, Vt)
    assert_grad_close(host_bf16_to_f64(dH), ref_dH, what="dH")
    vr = np.unique(np.concatenate([y, workloads.sample_rows(Vt, 40, seed=4), [Vt, V - 1]]))
    ref_dW = oracle_mod.backward_dw(d["h"], d["W"], y, g64, ref_lse, Vt, vrows=vr)
    assert_grad_close(dW[torch.from_numpy(vr).cuda()].cpu().numpy(), ref_dW, what="dW rows")
    # the same vocabulary as 8 shards merges to the same bits
    parts = torch.stack([rlk.linear_logp_fwd(h, W[a:a + n], yd, Vt, vocab_start=a, partial=True)
                         for a, n in rlk.shard_bounds(V, Vt, 8)])
    slogp, slse = rlk.lse_merge(parts)
    assert torch.equal(slogp, logp) and torch.equal(slse, lse)


def test_largest_hidden(rlk, oracle_mod):
    T, H, V, Vt = 3, MAX_HIDDEN, 1024, 1000
    d = workloads.make_inputs(workloads.Workload("maxh", T=T, H=H, V=V, V_true=Vt, seed=5))
    h, W, y, g = dev_bf16(d["h"]), dev_bf16(d["W"]), dev(d["y"]), dev(d["g"])
    logp, lse = rlk.linear_logp_fwd(h, W, y, Vt)
    dH, dW = rlk.linear_logp_bwd(h, W, y, lse, g, Vt)
    ref_logp, ref_lse = oracle_mod.forward(d["h"], d["W"], d["y"], Vt)
    assert_logp_close(logp.cpu().numpy(), ref_logp)
    g64 = d["g"].astype(np.float64)
    assert_grad_close(host_bf16_to_f64(dH), oracle_mod.backward_dh(d["h"], d["W"], d["y"], g64, Vt),
                      what="dH")
    assert_grad_close(dW.cpu().numpy(), oracle_mod.backward_dw(d["h"], d["W"], d["y"], g64, ref_lse, Vt),
                      what="dW")


def test_token_reduction_longer_than_one_accumulation_chunk(rlk, oracle_mod):
    # dW sums over the tokens; past 65536 tokens the tensor-core accumulator is restarted
    # and the chunk sums are folded in ascending order into the fp32 dW itself (the path
    # that keeps plain stores). 65536 + 300 tokens: one full chunk and a ragged one.
    T, H, V, Vt = 65536 + 300, 64, 512, 500
    d = workloads.make_inputs(workloads.Workload("longT", T=T, H=H, V=V, V_true=Vt, seed=6))
    h, W, y, g = dev_bf16(d["h"]), dev_bf16(d["W"]), dev(d["y"]), dev(d["g"])
    logp, lse = rlk.linear_logp_fwd(h, W, y, Vt)
    dH, dW = rlk.linear_logp_bwd(h, W, y, lse, g, Vt)
    torch.cuda.synchronize()
    ref_logp, ref_lse = oracle_mod.forward(d["h"], d["W"], d["y"], Vt)
    assert_logp_close(logp.cpu().numpy(), ref_logp)
    g64 = d["g"].astype(np.float64)
    ref_dW = oracle_mod.backward_dw(d["h"], d["W"], d["y"], g64, ref_lse, Vt)
    assert_grad_close(dW.cpu().numpy(), ref_dW, what="dW")
    assert torch.count_nonzero(dW[Vt:]).item() == 0
    rows = workloads.sample_rows(T, 64, seed=7)
    ref_dH = oracle_mod.backward_dh(d["h"], d["W"], d["y"], g64, Vt, rows=rows)
    assert_grad_close(host_bf16_to_f64(dH[torch.from_numpy(rows).cuda()]), ref_dH, what="dH rows")


def test_one_past_the_limits_is_rejected(rlk):
    lib = rlk.lib()
    import ctypes
    fake = ctypes.c_void_p(0x100000)
    st = lib.rlk_linear_logp_fwd(fake, fake, fake, 0, 64, MAX_VOCAB + 1, 0, MAX_VOCAB + 1, fake, fake,
                                 None, None, fake, 1 << 30, None)
    assert st == rlk.RLK_ERR_UNSUPPORTED
    st = lib.rlk_linear_logp_fwd(fake, fake, fake, 0, MAX_HIDDEN + 8, 1024, 0, 1024, fake, fake,
                                 None, None, fake, 1 << 30, None)
    assert st == rlk.RLK_ERR_UNSUPPORTED
