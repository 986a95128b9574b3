"""GPU vs fp64 oracle, element by element, on small and ragged shapes.

Every call goes through the C ABI (ctypes binding of librlk.so). Tolerances:
max |dlogp| <= 2e-3 nats and relative L2 <= 1e-2 for dH and dW.
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


def _inputs(T, H, V, Vt, seed):
    if (T, H, V, Vt) == (workloads.TINY.T, workloads.TINY.H, workloads.TINY.V, workloads.TINY.V_true):
        return workloads.make_inputs(workloads.TINY)   # the tiny workload, seed 0
    w = workloads.Workload("case", T=T, H=H, V=V, V_true=Vt, seed=seed)
    return workloads.make_inputs(w)


SHAPES = [
    # (T, H, V, V_true)
    (64, 256, 4096, 4096),      # the tiny workload
    (1, 64, 256, 256),          # one token, one tile
    (7, 136, 1100, 1030),       # second leaf holds 6 valid columns; K tail of 8
    (129, 200, 2500, 2345),     # ragged everything: T, H (K and N tails), V, V_true
    (300, 512, 20480, 20000),   # 20 leaves over 8 super-shards of 3
]


@pytest.mark.parametrize("T,H,V,Vt", SHAPES)
def test_forward_backward_parity(rlk, oracle_mod, T, H, V, Vt):
    d = _inputs(T, H, V, Vt, seed=T + H)
    h, W, y, g = dev_bf16(d["h"]), dev_bf16(d["W"]), dev(d["y"]), dev(d["g"])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    logp, lse = rlk.linear_logp_fwd(h, W, y, Vt, err_flag=err)
    dH, dW = rlk.linear_logp_bwd(h, W, y, lse, g, Vt, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0

    ref_logp, ref_lse = oracle_mod.forward(d["h"], d["W"], d["y"], Vt)
    assert_logp_close(logp.cpu().numpy(), ref_logp)
    assert_logp_close(lse.cpu().numpy(), ref_lse)

    g64 = d["g"].astype(np.float64)
    ref_dH = oracle_mod.backward_dh(d["h"], d["W"], d["y"], g64, Vt)
    ref_dW = oracle_mod.backward_dw(d["h"], d["W"], d["y"], g64, ref_lse, Vt)
    assert dH.dtype == torch.bfloat16 and dW.dtype == torch.float32
    assert_grad_close(host_bf16_to_f64(dH), ref_dH, what="dH")
    dW_h = dW.cpu().numpy()
    assert_grad_close(dW_h, ref_dW, what="dW")
    assert np.all(dW_h[Vt:] == 0.0)


def _scale_bf16(bits, k):
    """bf16 bits times 2**k: an exponent shift, exact for these magnitudes."""
    f = (bits.astype(np.uint32) << 16).view(np.float32) * np.float32(2.0 ** k)
    return workloads.bf16_bits(f)


def test_large_logit_range(rlk, oracle_mod):
    # h * 16 and W * 4 give logits of standard deviation ~20 (|z| up to ~100): a running max
    # or merge that did not shift by the maximum would overflow exp and give inf / NaN here.
    # Rows with g = 0 must get exactly zero dH rows.
    T, H, V, Vt = 129, 256, 2500, 2345
    d = _inputs(T, H, V, Vt, seed=77)
    hb, Wb = _scale_bf16(d["h"], 4), _scale_bf16(d["W"], 2)
    g = d["g"].copy()
    g[::7] = 0.0
    h, W, y, gd = dev_bf16(hb), dev_bf16(Wb), dev(d["y"]), dev(g)
    logp, lse = rlk.linear_logp_fwd(h, W, y, Vt)
    dH, dW = rlk.linear_logp_bwd(h, W, y, lse, gd, Vt)
    torch.cuda.synchronize()
    ref_logp, ref_lse = oracle_mod.forward(hb, Wb, d["y"], Vt)
    assert np.abs(ref_lse).max() > 40.0          # the range this test is meant to reach
    assert_logp_close(logp.cpu().numpy(), ref_logp)
    assert_logp_close(lse.cpu().numpy(), ref_lse)
    g64 = g.astype(np.float64)
    ref_dH = oracle_mod.backward_dh(hb, Wb, d["y"], g64, Vt)
    assert_grad_close(host_bf16_to_f64(dH), ref_dH, what="dH")
    ref_dW = oracle_mod.backward_dw(hb, Wb, d["y"], g64, ref_lse, Vt)
    assert_grad_close(dW.cpu().numpy(), ref_dW, what="dW")
    assert torch.count_nonzero(dH[::7]).item() == 0
    # the saved-logits pair gives the same bits; the saved bf16 probabilities stay within
    # tolerance (each probability is stored relative to its 64-column running maximum)
    (logp2, lse2), z = rlk.linear_logp_fwd_save(h, W, y, Vt)
    dH2, dW2 = rlk.linear_logp_bwd_saved(h, W, y, lse, gd, z, Vt)
    assert torch.equal(logp2, logp) and torch.equal(lse2, lse)
    assert torch.equal(dH2, dH) and torch.equal(dW2, dW)
    (logp3, lse3), pbuf = rlk.linear_logp_fwd_save_probs(h, W, y, Vt)
    dH3, dW3 = rlk.linear_logp_bwd_saved_probs(h, W, y, lse, gd, pbuf, Vt)
    assert torch.equal(logp3, logp) and torch.equal(lse3, lse)
    assert_grad_close(host_bf16_to_f64(dH3), ref_dH, what="dH (saved probs)")
    assert_grad_close(dW3.cpu().numpy(), ref_dW, what="dW (saved probs)")


def test_fp32_dH_partial_matches(rlk, oracle_mod):
    T, H, V, Vt = 96, 128, 3000, 2900
    d = _inputs(T, H, V, Vt, seed=5)
    h, W, y, g = dev_bf16(d["h"]), dev_bf16(d["W"]), dev(d["y"]), dev(d["g"])
    _, lse = rlk.linear_logp_fwd(h, W, y, Vt)
    dH32, _ = rlk.linear_logp_bwd(h, W, y, lse, g, Vt, dH_fp32_partial=True, want_dW=False)
    dH16, _ = rlk.linear_logp_bwd(h, W, y, lse, g, Vt, want_dW=False)
    assert dH32.dtype == torch.float32
    # the bf16 output is exactly the fp32 accumulator rounded once
    assert torch.equal(dH32.to(torch.bfloat16), dH16)
    ref_lse = oracle_mod.forward(d["h"], d["W"], d["y"], Vt)[1]
    ref = oracle_mod.backward_dh(d["h"], d["W"], d["y"], d["g"].astype(np.float64), Vt)
    assert_grad_close(dH32.cpu().numpy().astype(np.float64), ref, tol=5e-3, what="dH fp32")
    assert np.isfinite(ref_lse).all()


def test_invalid_targets_flag_nan_and_zero_grad(rlk, oracle_mod):
    T, H, V, Vt = 40, 64, 2048, 2000
    d = _inputs(T, H, V, Vt, seed=9)
    y = d["y"].copy()
    y[3] = -1
    y[17] = Vt          # padding column: not a valid target
    y[39] = V + 5
    h, W, yd, g = dev_bf16(d["h"]), dev_bf16(d["W"]), dev(y), dev(d["g"])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    logp, lse = rlk.linear_logp_fwd(h, W, yd, Vt, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & rlk.RLK_FLAG_BAD_TARGET
    lp = logp.cpu().numpy()
    bad = np.array([3, 17, 39])
    assert np.all(np.isnan(lp[bad]))
    good = np.setdiff1d(np.arange(T), bad)
    ref_logp, ref_lse = oracle_mod.forward(d["h"], d["W"], y, Vt)
    assert_logp_close(lp[good], ref_logp[good])
    assert_logp_close(lse.cpu().numpy(), ref_lse)     # lse stays defined for every row
    err.zero_()
    dH, dW = rlk.linear_logp_bwd(h, W, yd, lse, g, Vt, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & rlk.RLK_FLAG_BAD_TARGET
    assert torch.all(dH[bad].float() == 0)
    ref_dH = oracle_mod.backward_dh(d["h"], d["W"], y, d["g"].astype(np.float64), Vt)
    assert_grad_close(host_bf16_to_f64(dH), ref_dH, what="dH")
    ref_dW = oracle_mod.backward_dw(d["h"], d["W"], y, d["g"].astype(np.float64), ref_lse, Vt)
    assert_grad_close(dW.cpu().numpy(), ref_dW, what="dW")


def test_empty_batch_is_a_no_op(rlk):
    h = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((512, 64), dtype=torch.bfloat16, device="cuda")
    y = torch.empty(0, dtype=torch.int64, device="cuda")
    logp, lse = rlk.linear_logp_fwd(h, W, y, 500)
    dH, dW = rlk.linear_logp_bwd(h, W, y, lse, torch.empty(0, device="cuda"), 500, want_dW=False)
    assert logp.numel() == 0 and dH.numel() == 0


def test_closed_forms_on_gpu(rlk):
    # W = 0 (padding rows arbitrary): logp = -log V_true exactly up to fp32
    T, H, V, Vt = 130, 64, 3000, 2999
    W = torch.zeros((V, H), dtype=torch.bfloat16, device="cuda")
    W[Vt:] = 3.0
    h = torch.randn((T, H), device="cuda").to(torch.bfloat16)
    y = torch.randint(0, Vt, (T,), device="cuda")
    logp, lse = rlk.linear_logp_fwd(h, W, y, Vt)
    assert torch.allclose(logp, torch.full_like(logp, -np.log(Vt)), atol=2e-5, rtol=0)
    # V_true = 1: logp = 0 and zero gradients
    W1 = torch.randn((256, H), device="cuda").to(torch.bfloat16)
    y0 = torch.zeros(T, dtype=torch.int64, device="cuda")
    logp1, lse1 = rlk.linear_logp_fwd(h, W1, y0, 1)
    # exactly 0 up to fp32 rounding of z0 + log(e(z0 - z0)) (the fma residual of z0 log2 e)
    assert torch.all(logp1.abs() <= 1e-5)
    g = torch.randn(T, device="cuda")
    dH, dW = rlk.linear_logp_bwd(h, W1, y0, lse1, g, 1)
    assert dH.float().abs().max() <= 1e-4 and dW.abs().max() <= 1e-4
    assert torch.all(dW[1:] == 0)


@pytest.mark.parametrize("S,V,Vt", [(2, 20480, 20000), (4, 20480, 20000), (8, 24576, 24000)])
def test_sharded_forward_is_bitwise_unsharded(rlk, oracle_mod, S, V, Vt):
    T, H = 300, 512
    d = _inputs(T, H, V, Vt, seed=21)
    h, W, y, g = dev_bf16(d["h"]), dev_bf16(d["W"]), dev(d["y"]), dev(d["g"])
    logp, lse = rlk.linear_logp_fwd(h, W, y, Vt)
    bounds = rlk.shard_bounds(V, Vt, S)
    parts = torch.stack([rlk.linear_logp_fwd(h, W[a:a + n], y, Vt, vocab_start=a, partial=True)
                         for a, n in bounds])
    slogp, slse = rlk.lse_merge(parts)
    assert torch.equal(slogp, logp) and torch.equal(slse, lse)
    # each shard's statistics against the oracle's (compared as the shard's own lse)
    p = parts.cpu().numpy().astype(np.float64)
    for i, (a, n) in enumerate(bounds):
        m, s, zt = oracle_mod.shard_stats(d["h"], d["W"][a:a + n], d["y"], a, Vt)
        ok = s > 0
        assert np.array_equal(ok, p[i, :, 1] > 0)
        assert_logp_close(p[i, ok, 0] + np.log(p[i, ok, 1]), m[ok] + np.log(s[ok]))
        own = np.isfinite(zt)
        assert np.array_equal(own, np.isfinite(p[i, :, 2]))
        assert_logp_close(p[i, own, 2], zt[own])
    # backward per shard: dW rows are bitwise the unsharded rows; dH partials sum within tolerance
    dH, dW = rlk.linear_logp_bwd(h, W, y, lse, g, Vt)
    dH_parts = []
    for a, n in bounds:
        dHp, dWp = rlk.linear_logp_bwd(h, W[a:a + n], y, lse, g, Vt, vocab_start=a, dH_fp32_partial=True)
        assert torch.equal(dWp, dW[a:a + n])
        dH_parts.append(dHp)
    dH_s = rlk.shard_sum_bf16(torch.stack(dH_parts))
    ref_dH = oracle_mod.backward_dh(d["h"], d["W"], d["y"], d["g"].astype(np.float64), Vt)
    assert_grad_close(host_bf16_to_f64(dH_s), ref_dH, what="sharded dH")


def test_targets_on_tile_leaf_shard_and_vocab_boundaries(rlk, oracle_mod):
    # targets at the first and last column of 256-column tiles, 1024-column leaves, the last
    # valid column and the columns on both sides of every shard boundary of an 8-way split
    H, V, Vt = 192, 24576, 24000
    bounds = rlk.shard_bounds(V, Vt, 8)
    ys = {0, 1, 255, 256, 1023, 1024, 1025, Vt - 2, Vt - 1}
    for a, _ in bounds[1:]:
        ys |= {a - 1, a, a + 1}
    y_np = np.array(sorted(ys), dtype=np.int64)
    T = y_np.shape[0]
    d = _inputs(T, H, V, Vt, seed=91)
    h, W, y, g = dev_bf16(d["h"]), dev_bf16(d["W"]), dev(y_np), dev(d["g"])
    logp, lse = rlk.linear_logp_fwd(h, W, y, Vt)
    dH, dW = rlk.linear_logp_bwd(h, W, y, lse, g, Vt)
    torch.cuda.synchronize()
    ref_logp, ref_lse = oracle_mod.forward(d["h"], d["W"], y_np, Vt)
    assert_logp_close(logp.cpu().numpy(), ref_logp)
    g64 = d["g"].astype(np.float64)
    assert_grad_close(host_bf16_to_f64(dH), oracle_mod.backward_dh(d["h"], d["W"], y_np, g64, Vt), what="dH")
    assert_grad_close(dW.cpu().numpy(), oracle_mod.backward_dw(d["h"], d["W"], y_np, g64, ref_lse, Vt),
                      what="dW")
    # exactly one shard owns each target; the merged shards give the unsharded bits
    parts = torch.stack([rlk.linear_logp_fwd(h, W[a:a + n], y, Vt, vocab_start=a, partial=True)
                         for a, n in bounds])
    owners = torch.isfinite(parts[:, :, 2]).sum(dim=0)
    assert torch.all(owners == 1)
    slogp, slse = rlk.lse_merge(parts)
    assert torch.equal(slogp, logp) and torch.equal(slse, lse)


def test_lse_merge_against_oracle(rlk, oracle_mod):
    rng = np.random.default_rng(3)
    for S in (1, 2, 4, 8):
        T = 1000
        m = (rng.standard_normal((S, T)) * 4 + 10).astype(np.float32)
        s = rng.uniform(1.0, 5e4, (S, T)).astype(np.float32)
        zt = np.full((S, T), -np.inf, np.float32)
        owner = rng.integers(0, S, T)
        if S > 1:
            owner[:50] = 0
            m[1, :50] = -np.inf      # shard 1 is empty for the first 50 tokens
            s[1, :50] = 0.0
        zt[owner, np.arange(T)] = (m[owner, np.arange(T)] - rng.uniform(0, 8, T)).astype(np.float32)
        parts = np.stack([m, s, zt], axis=-1)
        logp, lse = rlk.lse_merge(dev(parts))
        rl, rs = oracle_mod.lse_merge(m.astype(np.float64), s.astype(np.float64), zt.astype(np.float64))
        np.testing.assert_allclose(lse.cpu().numpy(), rs, rtol=0, atol=2e-5)
        np.testing.assert_allclose(logp.cpu().numpy(), rl, rtol=0, atol=4e-5)


def test_shard_sum_bf16(rlk):
    for n in (1, 7, 4096, 4099):
        p = torch.randn((3, n), device="cuda")
        out = rlk.shard_sum_bf16(p)
        ref = ((p[0] + p[1]) + p[2]).to(torch.bfloat16)
        assert torch.equal(out, ref)


@pytest.mark.parametrize("T,H,V,Vt", [(300, 512, 20480, 20000), (129, 200, 2500, 2345), (1, 64, 256, 256)])
def test_saved_logits_path_is_bitwise_the_recompute_path(rlk, T, H, V, Vt):
    d = _inputs(T, H, V, Vt, seed=T * 7 + 1)
    h, W, y, g = dev_bf16(d["h"]), dev_bf16(d["W"]), dev(d["y"]), dev(d["g"])
    logp, lse = rlk.linear_logp_fwd(h, W, y, Vt)
    (logp2, lse2), z = rlk.linear_logp_fwd_save(h, W, y, Vt)
    assert torch.equal(logp, logp2) and torch.equal(lse, lse2)
    dH, dW = rlk.linear_logp_bwd(h, W, y, lse, g, Vt)
    dH2, dW2 = rlk.linear_logp_bwd_saved(h, W, y, lse, g, z, Vt)
    assert torch.equal(dH, dH2) and torch.equal(dW, dW2)
    # the saved logits are the fp32 products h W^T of the valid columns
    ref = host_bf16_to_f64(h) @ host_bf16_to_f64(W).T
    got = z[:, :Vt].cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(got, ref[:, :Vt], rtol=0, atol=1e-4 * max(1.0, np.abs(ref).max()))


def test_saved_logits_sharded_and_invalid_targets(rlk):
    T, H, V, Vt = 300, 512, 20480, 20000
    d = _inputs(T, H, V, Vt, seed=77)
    yb = d["y"].copy()
    yb[[5, 200]] = [-3, Vt + 1]
    h, W, y, g = dev_bf16(d["h"]), dev_bf16(d["W"]), dev(yb), dev(d["g"])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    logp, lse = rlk.linear_logp_fwd(h, W, y, Vt)
    dH, dW = rlk.linear_logp_bwd(h, W, y, lse, g, Vt)
    for a, n in rlk.shard_bounds(V, Vt, 2):
        _, z = rlk.linear_logp_fwd_save(h, W[a:a + n], y, Vt, vocab_start=a, partial=True)
        dHp, dWp = rlk.linear_logp_bwd_saved(h, W[a:a + n], y, lse, g, z, Vt, vocab_start=a,
                                             dH_fp32_partial=True, err_flag=err)
        assert torch.equal(dWp, dW[a:a + n])
        assert torch.all(dHp[[5, 200]] == 0)
    torch.cuda.synchronize()
    assert int(err.item()) & rlk.RLK_FLAG_BAD_TARGET


@pytest.mark.parametrize("T,H,V,Vt", [(300, 512, 20480, 20000), (129, 200, 2500, 2345), (64, 256, 4096, 4096)])
def test_saved_probs_path(rlk, oracle_mod, T, H, V, Vt):
    """bf16 saved probabilities: logp / lse bit-identical to the plain forward, gradients
    within the tolerance of the oracle (not bitwise: p carries one bf16 rounding)."""
    d = _inputs(T, H, V, Vt, seed=T * 3 + 2)
    h, W, y, g = dev_bf16(d["h"]), dev_bf16(d["W"]), dev(d["y"]), dev(d["g"])
    logp, lse = rlk.linear_logp_fwd(h, W, y, Vt)
    (logp2, lse2), pbuf = rlk.linear_logp_fwd_save_probs(h, W, y, Vt)
    assert torch.equal(logp, logp2) and torch.equal(lse, lse2)
    dH, dW = rlk.linear_logp_bwd_saved_probs(h, W, y, lse, g, pbuf, Vt)
    ref_lse = oracle_mod.forward(d["h"], d["W"], d["y"], Vt)[1]
    g64 = d["g"].astype(np.float64)
    ref_dH = oracle_mod.backward_dh(d["h"], d["W"], d["y"], g64, Vt)
    ref_dW = oracle_mod.backward_dw(d["h"], d["W"], d["y"], g64, ref_lse, Vt)
    assert_grad_close(host_bf16_to_f64(dH), ref_dH, what="dH (saved probs)")
    assert_grad_close(dW.cpu().numpy(), ref_dW, what="dW (saved probs)")
    assert torch.all(dW[Vt:] == 0)
    # sharded: each shard's probabilities give its dW rows
    for a, n in rlk.shard_bounds(V, Vt, 2) if V >= 20480 else []:
        _, pb = rlk.linear_logp_fwd_save_probs(h, W[a:a + n], y, Vt, vocab_start=a, partial=True)
        _, dWp = rlk.linear_logp_bwd_saved_probs(h, W[a:a + n], y, lse, g, pb, Vt, vocab_start=a,
                                                 want_dH=False)
        assert_grad_close(dWp.cpu().numpy(), ref_dW[a:a + n], what="shard dW (saved probs)")


def test_dH_large_batch_sampled_rows_and_sub_batch(rlk, oracle_mod):
    # dH at T = 8192, H = 2048 (32 row tiles x 8 column tiles: several waves of work items over
    # the resident CTA pairs): sampled rows against the oracle, and every row of a 512-row
    # sub-batch (2 x 8 items, all in the first wave) bit for bit against the same rows of the
    # full batch, in bf16 and as the fp32 shard partial.
    T, H, V, Vt = 8192, 2048, 20480, 20000
    d = _inputs(T, H, V, Vt, seed=88)
    h, W, y, g = dev_bf16(d["h"]), dev_bf16(d["W"]), dev(d["y"]), dev(d["g"])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    logp, lse = rlk.linear_logp_fwd(h, W, y, Vt, err_flag=err)
    dH, _ = rlk.linear_logp_bwd(h, W, y, lse, g, Vt, want_dW=False, err_flag=err)
    dHp, _ = rlk.linear_logp_bwd(h, W, y, lse, g, Vt, want_dW=False, dH_fp32_partial=True)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rows = np.concatenate([np.arange(0, T, 331), np.arange(4860, 4870), [T - 1]])
    g64 = d["g"].astype(np.float64)
    ref = oracle_mod.backward_dh(d["h"], d["W"], d["y"], g64, Vt, rows=rows)
    assert_grad_close(host_bf16_to_f64(dH)[rows], ref, what="dH")
    assert_grad_close(dHp.cpu().numpy()[rows], ref, what="dH fp32")
    lo = 4608
    sub = slice(lo, lo + 512)
    hs, ys, gs, ls = h[sub].contiguous(), y[sub].contiguous(), g[sub].contiguous(), lse[sub].contiguous()
    dHs, _ = rlk.linear_logp_bwd(hs, W, ys, ls, gs, Vt, want_dW=False)
    dHps, _ = rlk.linear_logp_bwd(hs, W, ys, ls, gs, Vt, want_dW=False, dH_fp32_partial=True)
    torch.cuda.synchronize()
    assert torch.equal(dHs, dH[sub])
    assert torch.equal(dHps, dHp[sub])
