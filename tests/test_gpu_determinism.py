"""Bitwise properties of the GPU path (difference exactly zero, no tolerance):
run-to-run determinism, independence from the stream and from concurrent
work, and batch invariance (a token's logp, lse and dH rows do not depend on
the batch it sits in or on its row inside the batch)."""
import numpy as np
import pytest
import torch

import workloads
from gpu_util import assert_logp_close, dev, dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rlk():
    from deterministic_token_logprob_gb300 import build
    build.build()
    import deterministic_token_logprob_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def _mid():
    w = workloads.Workload("mid", T=700, H=512, V=9000, V_true=8999, seed=31)
    d = workloads.make_inputs(w)
    return w, d, dev_bf16(d["h"]), dev_bf16(d["W"]), dev(d["y"]), dev(d["g"])


def _all_outputs(rlk, w, h, W, y, g, stream=None):
    logp, lse = rlk.linear_logp_fwd(h, W, y, w.V_true, stream=stream)
    dH, dW = rlk.linear_logp_bwd(h, W, y, lse, g, w.V_true, stream=stream)
    return logp, lse, dH, dW


def test_run_to_run_bitwise(rlk):
    w, d, h, W, y, g = _mid()
    first = _all_outputs(rlk, w, h, W, y, g)
    for _ in range(3):
        again = _all_outputs(rlk, w, h, W, y, g)
        for a, b in zip(first, again):
            assert torch.equal(a, b)


def test_stream_and_concurrent_work_do_not_change_bits(rlk):
    w, d, h, W, y, g = _mid()
    ref = _all_outputs(rlk, w, h, W, y, g)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        got = _all_outputs(rlk, w, h, W, y, g, stream=side)
    side.synchronize()
    for a, b in zip(ref, got):
        assert torch.equal(a, b)
    # the same call while another stream keeps the SMs busy with a large GEMM
    busy = torch.cuda.Stream()
    x = torch.randn((8192, 8192), device="cuda", dtype=torch.bfloat16)
    torch.cuda.synchronize()
    with torch.cuda.stream(busy):
        for _ in range(4):
            x = (x @ x).clamp_(-1, 1)
    got = _all_outputs(rlk, w, h, W, y, g)
    torch.cuda.synchronize()
    for a, b in zip(ref, got):
        assert torch.equal(a, b)


def test_two_calls_running_at_once_on_two_streams(rlk):
    # Each call hands out its work items from a counter in its own workspace; two calls whose
    # kernels overlap on the GPU (so neither has all SMs) must not disturb each other.
    w, d, h, W, y, g = _mid()
    ref = _all_outputs(rlk, w, h, W, y, g)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [[], []]
    for rep in range(3):
        for i, st in enumerate(streams):
            with torch.cuda.stream(st):
                outs[i].append(_all_outputs(rlk, w, h, W, y, g, stream=st))
    torch.cuda.synchronize()
    for per_stream in outs:
        for got in per_stream:
            for a, b in zip(ref, got):
                assert torch.equal(a, b)


@pytest.mark.parametrize("shape", [(700, 512, 9000, 8999), (300, 256, 70000, 69000)])
def test_backward_stages_match_one_call(rlk, shape):
    # The backward launched stage by stage (dz, then dH, then dW, sharing one workspace) gives
    # the bits of one rlk_linear_logp_bwd call; so do dH and dW launched on two streams at once
    # after dz. The second shape's dH reduces over more than one 65536-column chunk (fp32
    # running sum in the workspace).
    T, H, V, Vt = shape
    w = workloads.Workload("stages", T=T, H=H, V=V, V_true=Vt, seed=33)
    d = workloads.make_inputs(w)
    h, W, y, g = dev_bf16(d["h"]), dev_bf16(d["W"]), dev(d["y"]), dev(d["g"])
    _, lse = rlk.linear_logp_fwd(h, W, y, Vt)
    for partial in (False, True):
        ref_dH, ref_dW = rlk.linear_logp_bwd(h, W, y, lse, g, Vt, dH_fp32_partial=partial)
        ws = torch.empty(rlk.bwd_workspace_bytes(T, H, V), dtype=torch.uint8, device="cuda")
        dH = torch.full_like(ref_dH, float("nan"))
        dW = torch.full_like(ref_dW, float("nan"))
        out = (dH, dW)
        rlk.linear_logp_bwd(h, W, y, lse, g, Vt, dH_fp32_partial=partial, out=out, workspace=ws,
                            stages=rlk.RLK_BWD_DZ)
        rlk.linear_logp_bwd(h, W, y, lse, g, Vt, dH_fp32_partial=partial, out=out, workspace=ws,
                            stages=rlk.RLK_BWD_DH)
        rlk.linear_logp_bwd(h, W, y, lse, g, Vt, dH_fp32_partial=partial, out=out, workspace=ws,
                            stages=rlk.RLK_BWD_DW)
        torch.cuda.synchronize()
        assert torch.equal(dH, ref_dH) and torch.equal(dW, ref_dW)
        # dH and dW at the same time on two streams, both after the dz stage
        dH.fill_(float("nan"))
        dW.fill_(float("nan"))
        rlk.linear_logp_bwd(h, W, y, lse, g, Vt, dH_fp32_partial=partial, out=out, workspace=ws,
                            stages=rlk.RLK_BWD_DZ)
        dz_done = torch.cuda.Event()
        dz_done.record()
        side = torch.cuda.Stream()
        side.wait_event(dz_done)
        with torch.cuda.stream(side):
            rlk.linear_logp_bwd(h, W, y, lse, g, Vt, dH_fp32_partial=partial, out=out, workspace=ws,
                                stages=rlk.RLK_BWD_DW, stream=side)
        rlk.linear_logp_bwd(h, W, y, lse, g, Vt, dH_fp32_partial=partial, out=out, workspace=ws,
                            stages=rlk.RLK_BWD_DH)
        torch.cuda.synchronize()
        assert torch.equal(dH, ref_dH) and torch.equal(dW, ref_dW)


def test_backward_stages_per_vocab_shard(rlk):
    # the staged backward of each shard of a 2-way split (fp32 dH partials, the shard's dW
    # rows) equals that shard's one-call backward bit for bit, as the sharded bench step uses it
    T, H, V, Vt = 300, 256, 70000, 69000
    w = workloads.Workload("stages_shard", T=T, H=H, V=V, V_true=Vt, seed=34)
    d = workloads.make_inputs(w)
    h, W, y, g = dev_bf16(d["h"]), dev_bf16(d["W"]), dev(d["y"]), dev(d["g"])
    _, lse = rlk.linear_logp_fwd(h, W, y, Vt)
    for a, n in rlk.shard_bounds(V, Vt, 2):
        Ws = W[a:a + n]
        ref_dH, ref_dW = rlk.linear_logp_bwd(h, Ws, y, lse, g, Vt, vocab_start=a, dH_fp32_partial=True)
        ws = torch.empty(rlk.bwd_workspace_bytes(T, H, n), dtype=torch.uint8, device="cuda")
        dH = torch.full_like(ref_dH, float("nan"))
        dW = torch.full_like(ref_dW, float("nan"))
        for st in (rlk.RLK_BWD_DZ, rlk.RLK_BWD_DH, rlk.RLK_BWD_DW):
            rlk.linear_logp_bwd(h, Ws, y, lse, g, Vt, vocab_start=a, dH_fp32_partial=True,
                                out=(dH, dW), workspace=ws, stages=st)
        torch.cuda.synchronize()
        assert torch.equal(dH, ref_dH) and torch.equal(dW, ref_dW), a


def _invariance(rlk, H, V, Vt, W_bits, W_dev, Ts, oracle_mod=None, check_dH=True):
    th, ty = workloads.invariance_targets(0, H=H, V_true=Vt)
    n = th.shape[0]
    g_target = np.linspace(-1.0, 1.0, n).astype(np.float32)   # fixed per-target upstream gradient
    seen_logp = {}
    seen_dH = {}
    for T in Ts:
        logp_t = np.full(n, np.nan, np.float32)
        lse_t = np.full(n, np.nan, np.float32)
        dH_t = np.zeros((n, H), np.float32) if check_dH else None
        for rep in range(2):
            for b in workloads.invariance_batches(T, 0, H=H, V_true=Vt):
                g = np.random.default_rng(T).standard_normal(T).astype(np.float32)
                g[b.target_rows] = g_target[b.target_ids]
                hd, yd, gd = dev_bf16(b.h), dev(b.y), dev(g)
                logp, lse = rlk.linear_logp_fwd(hd, W_dev, yd, Vt)
                lp = logp.cpu().numpy()[b.target_rows]
                ls = lse.cpu().numpy()[b.target_rows]
                if rep == 0:
                    logp_t[b.target_ids] = lp
                    lse_t[b.target_ids] = ls
                else:
                    assert np.array_equal(logp_t[b.target_ids].view(np.uint32), lp.view(np.uint32))
                if check_dH and rep == 0:
                    dH, _ = rlk.linear_logp_bwd(hd, W_dev, yd, lse, gd, Vt, want_dW=False,
                                                dH_fp32_partial=True)
                    dH_t[b.target_ids] = dH.cpu().numpy()[b.target_rows]
        assert not np.isnan(logp_t).any()
        seen_logp[T] = (logp_t, lse_t)
        seen_dH[T] = dH_t
    T0 = Ts[0]
    for T in Ts[1:]:
        assert np.array_equal(seen_logp[T][0].view(np.uint32), seen_logp[T0][0].view(np.uint32)), T
        assert np.array_equal(seen_logp[T][1].view(np.uint32), seen_logp[T0][1].view(np.uint32)), T
        if check_dH:
            assert np.array_equal(seen_dH[T].view(np.uint32), seen_dH[T0].view(np.uint32)), T
    if oracle_mod is not None:
        pick = np.arange(0, n, max(1, n // 8))
        ref_logp, _ = oracle_mod.forward(th[pick], W_bits, ty[pick], Vt)
        assert_logp_close(seen_logp[T0][0][pick], ref_logp)


def test_batch_invariance_small(rlk, oracle_mod):
    H, V, Vt = 256, 4096, 4000
    W_bits = workloads.make_W(V, H, 7)
    _invariance(rlk, H, V, Vt, W_bits, dev_bf16(W_bits), workloads.INVARIANCE_T, oracle_mod)


def test_row_position_inside_tile_does_not_matter(rlk):
    # one token placed at every row of a 128-row tile (and the next tile) gives one bit pattern
    H, V, Vt = 128, 2048, 2048
    W = dev_bf16(workloads.make_W(V, H, 3))
    one = workloads.make_h(1, H, 4)
    T = 300
    h = np.repeat(one, T, axis=0)
    y = np.full(T, 77, np.int64)
    logp, lse = rlk.linear_logp_fwd(dev_bf16(h), W, dev(y), Vt)
    lp = logp.cpu().numpy()
    assert np.all(lp.view(np.uint32) == lp[0].view(np.uint32))
