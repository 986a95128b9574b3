"""FP8 (E4M3, one power-of-two scale per row) LM head on the GPU against the oracle.

The quantizer is byte work: its codes and scales must equal the oracle's bit for
bit. The FP8 forward is compared with the oracle evaluated on the oracle's own
quantization of the same bf16 inputs (max |dlogp| <= 2e-3 nats), and the
straight-through backward with the oracle's straight-through gradients (relative
L2 <= 1e-2). Batch and shard invariance are bitwise, as for the bf16 path.
"""
import numpy as np
import pytest
import torch

import workloads
from gpu_util import (assert_grad_close, assert_logp_close, dev, dev_bf16, host_bf16_to_f64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rlk():
    from deterministic_token_logprob_gb300 import build
    build.build()
    import deterministic_token_logprob_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def _assert_quant_equal(rlk, oracle_mod, bits):
    x = dev_bf16(bits)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q, s = rlk.quantize_rows_e4m3(x, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rq, rs = oracle_mod.quantize_rows_e4m3(bits)
    np.testing.assert_array_equal(q.cpu().numpy(), rq)
    np.testing.assert_array_equal(s.cpu().numpy().astype(np.float64), rs)
    return q, s, (rq, rs)


def _quant_rows(rng, rows, cols):
    """Rows spanning the scale range: normal values times a per-row power of two from
    2^-125 (the two-factor path of 2^-e) to 2^100, an all-zero row, a row of exact
    midpoints between E4M3 neighbours (ties), and one with bf16 subnormals and -0."""
    x = rng.standard_normal((rows, cols)) * np.exp2(rng.integers(-125, 100, rows))[:, None]
    x[0] = 0.0
    if rows > 2 and cols >= 8:
        mids = np.array([1.125 + 0.0625, 3.25 + 0.125, 0.015625 * 1.5, 2.0 ** -9 * 1.5,
                         -(1.125 + 0.0625), 240.0 + 8.0, -(2.0 ** -8 * 1.5)])
        x[1] = 0.0
        x[1, 0] = 448.0
        x[1, 1:1 + len(mids)] = mids[:cols - 1]
    if rows > 3:
        x[2] = rng.standard_normal(cols) * 2.0 ** -130      # bf16 subnormals
        x[2, -1] = -0.0
    return workloads.bf16_bits(x.astype(np.float32))


# 4096 and 2048 columns take the one-pass kernel (rows held in registers), the others the
# general two-pass kernel (vector and scalar paths)
@pytest.mark.parametrize("rows,cols", [(37, 64), (5, 24), (9, 4096), (11, 2048), (3, 8), (1, 16),
                                       (70, 2064)])
def test_quantize_bit_exact(rlk, oracle_mod, rows, cols):
    rng = np.random.default_rng(rows * 1000 + cols)
    _assert_quant_equal(rlk, oracle_mod, _quant_rows(rng, rows, cols))


@pytest.mark.parametrize("cols", [32, 2048, 4096])
def test_quantize_non_finite_row_is_flagged(rlk, cols):
    x = np.ones((4, cols), np.float32)
    x[2, 5] = np.inf
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q, s = rlk.quantize_rows_e4m3(dev_bf16(workloads.bf16_bits(x)), err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == rlk.RLK_FLAG_NONFINITE
    s = s.cpu().numpy()
    assert np.isnan(s[2]) and np.all(q[2].cpu().numpy() == 0)
    assert np.all(s[[0, 1, 3]] == 2.0 ** -8)     # 1 <= 448 * 2^-8 and 1 > 448 * 2^-9


def _fp8_inputs(rlk, oracle_mod, T, H, V, Vt, seed):
    w = workloads.Workload("fp8", T=T, H=H, V=V, V_true=Vt, seed=seed)
    d = workloads.make_inputs(w)
    hq, hs, ohq = _assert_quant_equal(rlk, oracle_mod, d["h"])
    Wq, Ws, oWq = _assert_quant_equal(rlk, oracle_mod, d["W"])
    return d, (hq, hs, Wq, Ws), (ohq, oWq)


FP8_SHAPES = [
    # (T, H, V, V_true)
    (64, 256, 4096, 4096),      # the tiny workload's shape
    (1, 64, 256, 256),          # one token, one tile, half a K block
    (7, 144, 1100, 1030),       # K tail of 16 after one 128-element block
    (129, 208, 2500, 2345),     # ragged T, K, V, V_true
    (300, 512, 20480, 20000),   # 20 leaves over 8 super-shards
]


@pytest.mark.parametrize("T,H,V,Vt", FP8_SHAPES)
def test_fp8_forward_and_ste_backward_parity(rlk, oracle_mod, T, H, V, Vt):
    d, (hq, hs, Wq, Ws), (ohq, oWq) = _fp8_inputs(rlk, oracle_mod, T, H, V, Vt, seed=T + H + 1)
    y, g = dev(d["y"]), dev(d["g"])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    logp, lse = rlk.linear_logp_fwd_fp8(hq, hs, Wq, Ws, y, Vt, err_flag=err)
    h, W = dev_bf16(d["h"]), dev_bf16(d["W"])
    dH, dW = rlk.linear_logp_bwd_fp8(h, W, hq, hs, Wq, Ws, y, lse, g, Vt, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0

    ref_logp, ref_lse = oracle_mod.forward(ohq, oWq, d["y"], Vt)
    assert_logp_close(logp.cpu().numpy(), ref_logp)
    assert_logp_close(lse.cpu().numpy(), ref_lse)
    g64 = d["g"].astype(np.float64)
    ref_dH = oracle_mod.backward_dh_ste(ohq, oWq, d["h"], d["W"], d["y"], g64, Vt)
    ref_dW = oracle_mod.backward_dw_ste(ohq, oWq, d["h"], d["y"], g64, ref_lse, Vt)
    assert_grad_close(host_bf16_to_f64(dH), ref_dH, what="dH")
    assert_grad_close(dW.cpu().numpy(), ref_dW, what="dW")
    assert torch.all(dW[Vt:] == 0)
    # the quantized logits differ from the bf16 ones: the FP8 result is its own, not the bf16 path's
    b_logp, _ = rlk.linear_logp_fwd(h, W, y, Vt)
    assert not torch.equal(b_logp, logp) or T * Vt < 2


def test_fp8_shards_and_batches_bitwise(rlk, oracle_mod):
    T, H, V, Vt = 200, 256, 24576, 24000
    d, (hq, hs, Wq, Ws), _ = _fp8_inputs(rlk, oracle_mod, T, H, V, Vt, seed=5)
    y = dev(d["y"])
    logp, lse = rlk.linear_logp_fwd_fp8(hq, hs, Wq, Ws, y, Vt)
    for S in (2, 4, 8):
        parts = torch.stack([rlk.linear_logp_fwd_fp8(hq, hs, Wq[a:a + n], Ws[a:a + n], y, Vt,
                                                     vocab_start=a, partial=True)
                             for a, n in rlk.shard_bounds(V, Vt, S)])
        slogp, slse = rlk.lse_merge(parts)
        assert torch.equal(slogp, logp) and torch.equal(slse, lse), S
    # batch invariance: the same rows inside other batches (quantized per row, so the
    # codes of a token do not depend on its batch either)
    h = dev_bf16(d["h"])
    for lo, hi in ((0, 1), (3, 10), (17, 200), (150, 200)):
        q2, s2 = rlk.quantize_rows_e4m3(h[lo:hi].contiguous())
        assert torch.equal(q2, hq[lo:hi]) and torch.equal(s2, hs[lo:hi])
        l2, e2 = rlk.linear_logp_fwd_fp8(q2, s2, Wq, Ws, y[lo:hi].contiguous(), Vt)
        assert torch.equal(l2, logp[lo:hi]) and torch.equal(e2, lse[lo:hi]), (lo, hi)
    # run to run
    l3, e3 = rlk.linear_logp_fwd_fp8(hq, hs, Wq, Ws, y, Vt)
    assert torch.equal(l3, logp) and torch.equal(e3, lse)


def test_fp8_closed_form_identical_rows(rlk):
    """Identical W rows quantize identically, so every logit of a token is equal and
    logp = -log V_true exactly up to fp32 rounding."""
    T, H, V, Vt = 33, 128, 3000, 2900
    rng = np.random.default_rng(3)
    row = rng.standard_normal(H).astype(np.float32) * 0.02
    W = dev_bf16(workloads.bf16_bits(np.tile(row, (V, 1))))
    h = dev_bf16(workloads.bf16_bits(rng.standard_normal((T, H)).astype(np.float32)))
    y = dev(rng.integers(0, Vt, T))
    hq, hs = rlk.quantize_rows_e4m3(h)
    Wq, Ws = rlk.quantize_rows_e4m3(W)
    logp, _ = rlk.linear_logp_fwd_fp8(hq, hs, Wq, Ws, y, Vt)
    np.testing.assert_allclose(logp.cpu().numpy(), -np.log(Vt), rtol=0, atol=2e-5)


def test_qwen3_8b_fp8_full_size_sampled(rlk, oracle_mod):
    """Qwen3-8B shape: the GPU's codes of all of W equal the oracle's; sampled tokens'
    logp against the oracle on the oracle's quantization; sampled straight-through dH
    rows and dW rows against the oracle (sparse g)."""
    w = workloads.QWEN3_8B
    W_bits = workloads.make_W(w.V, w.H, 0)
    d = workloads.make_inputs(w, with_W=False)
    h, W = dev_bf16(d["h"]), dev_bf16(W_bits)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    Wq, Ws = rlk.quantize_rows_e4m3(W, err_flag=err)
    hq, hs = rlk.quantize_rows_e4m3(h, err_flag=err)
    oWq = oracle_mod.quantize_rows_e4m3(W_bits)
    ohq = oracle_mod.quantize_rows_e4m3(d["h"])
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(Wq.cpu().numpy(), oWq[0]) and np.array_equal(Ws.cpu().numpy(), oWq[1])
    assert np.array_equal(hq.cpu().numpy(), ohq[0]) and np.array_equal(hs.cpu().numpy(), ohq[1])

    g, pos = workloads.sparse_g(w.T, 48, seed=12)
    y = dev(d["y"])
    logp, lse = rlk.linear_logp_fwd_fp8(hq, hs, Wq, Ws, y, w.V_true, err_flag=err)
    dH, dW = rlk.linear_logp_bwd_fp8(h, W, hq, hs, Wq, Ws, y, lse, dev(g), w.V_true, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref_logp, ref_lse = oracle_mod.forward(ohq, oWq, d["y"], w.V_true, rows=pos)
    assert_logp_close(logp.cpu().numpy()[pos], ref_logp)
    lse_full = np.full(w.T, np.nan)
    lse_full[pos] = ref_lse
    g64 = g.astype(np.float64)
    rows = pos[:12]
    ref_dH = oracle_mod.backward_dh_ste(ohq, oWq, d["h"], W_bits, d["y"], g64, w.V_true, rows=rows)
    assert_grad_close(host_bf16_to_f64(dH)[rows], ref_dH, what="dH rows")
    vr = np.array(sorted(set(workloads.sample_rows(w.V_true, 20, seed=13)) | set(d["y"][pos[:6]])
                         | {w.V_true, w.V - 1}), dtype=np.int64)
    ref_dW = oracle_mod.backward_dw_ste(ohq, oWq, d["h"], d["y"], g64, lse_full, w.V_true, vrows=vr)
    assert_grad_close(dW.cpu().numpy()[vr], ref_dW, what="dW rows")


def test_fp8_batch_invariance_full(rlk, oracle_mod):
    """128 fixed targets inside ragged batches T in {1, 7, 128, 1000, 4097} at the Qwen3-8B
    shape, FP8 path: each batch is quantized on the GPU (per-row scales, so a target's codes
    never depend on its batch); logp, lse and straight-through dH rows bitwise equal across T."""
    H, V, Vt = 4096, 151936, 151669
    W_bits = workloads.make_W(V, H, 0)
    W = dev_bf16(W_bits)
    Wq, Ws = rlk.quantize_rows_e4m3(W)
    th, ty = workloads.invariance_targets(0, H=H, V_true=Vt)
    n = th.shape[0]
    g_target = np.linspace(-1.0, 1.0, n).astype(np.float32)
    seen = {}
    for T in workloads.INVARIANCE_T:
        logp_t = np.full(n, np.nan, np.float32)
        lse_t = np.full(n, np.nan, np.float32)
        dH_t = np.zeros((n, H), np.float32)
        for b in workloads.invariance_batches(T, 0, H=H, V_true=Vt):
            g = np.random.default_rng(T).standard_normal(T).astype(np.float32)
            g[b.target_rows] = g_target[b.target_ids]
            hd, yd, gd = dev_bf16(b.h), dev(b.y), dev(g)
            hq, hs = rlk.quantize_rows_e4m3(hd)
            logp, lse = rlk.linear_logp_fwd_fp8(hq, hs, Wq, Ws, yd, Vt)
            dH, _ = rlk.linear_logp_bwd_fp8(hd, W, hq, hs, Wq, Ws, yd, lse, gd, Vt, want_dW=False,
                                            dH_fp32_partial=True)
            logp_t[b.target_ids] = logp.cpu().numpy()[b.target_rows]
            lse_t[b.target_ids] = lse.cpu().numpy()[b.target_rows]
            dH_t[b.target_ids] = dH.cpu().numpy()[b.target_rows]
        assert not np.isnan(logp_t).any()
        seen[T] = (logp_t, lse_t, dH_t)
    T0 = workloads.INVARIANCE_T[0]
    for T in workloads.INVARIANCE_T[1:]:
        for a, b in zip(seen[T], seen[T0]):
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), T
    pick = np.arange(0, n, 16)
    ohq = oracle_mod.quantize_rows_e4m3(th[pick])
    oWq = oracle_mod.quantize_rows_e4m3(W_bits)
    ref_logp, _ = oracle_mod.forward(ohq, oWq, ty[pick], Vt)
    assert_logp_close(seen[T0][0][pick], ref_logp)


def test_qwen3_30b_tp2_fp8_sharded(rlk, oracle_mod):
    """The 30B shape (T = 16384, H = 2048) in its two vocab shards on the FP8 path: merged
    shard statistics bitwise equal to the unsharded FP8 forward; sampled tokens against the
    oracle; sharded straight-through dH (fp32 partials, fixed-order sum) against the unsharded."""
    w = workloads.QWEN3_30B_TP2
    W_bits = workloads.make_W(w.V, w.H, 0)
    W = dev_bf16(W_bits)
    d = workloads.make_inputs(w, with_W=False)
    h, y = dev_bf16(d["h"]), dev(d["y"])
    hq, hs = rlk.quantize_rows_e4m3(h)
    Wq, Ws = rlk.quantize_rows_e4m3(W)
    logp, lse = rlk.linear_logp_fwd_fp8(hq, hs, Wq, Ws, y, w.V_true)
    parts = torch.stack([rlk.linear_logp_fwd_fp8(hq, hs, Wq[a:a + n], Ws[a:a + n], y, w.V_true,
                                                 vocab_start=a, partial=True)
                         for a, n in w.shards])
    slogp, slse = rlk.lse_merge(parts)
    assert torch.equal(slogp, logp) and torch.equal(slse, lse)
    rows = workloads.sample_rows(w.T, 12, seed=14)
    ref_logp, _ = oracle_mod.forward(oracle_mod.quantize_rows_e4m3(d["h"][rows]),
                                     oracle_mod.quantize_rows_e4m3(W_bits), d["y"][rows], w.V_true)
    assert_logp_close(slogp.cpu().numpy()[rows], ref_logp)
    g = dev(d["g"])
    dH_full, _ = rlk.linear_logp_bwd_fp8(h, W, hq, hs, Wq, Ws, y, lse, g, w.V_true, want_dW=False)
    dH_parts = torch.stack([
        rlk.linear_logp_bwd_fp8(h, W[a:a + n], hq, hs, Wq[a:a + n], Ws[a:a + n], y, slse, g,
                                w.V_true, vocab_start=a, dH_fp32_partial=True, want_dW=False)[0]
        for a, n in w.shards])
    dH = rlk.shard_sum_bf16(dH_parts)
    from gpu_util import rel_l2
    e = rel_l2(host_bf16_to_f64(dH), host_bf16_to_f64(dH_full))
    assert e <= 1e-2, e
