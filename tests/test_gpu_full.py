"""Full-size checks at the Qwen3 output-layer shapes, through the same C-ABI
calls and launch configuration the benchmark times.

The oracle cannot evaluate every output at these sizes, so the tests compare
sampled outputs it computes one by one (logp / dH rows of sampled tokens, dW
rows of sampled vocab rows; g is made sparse so that the dW rows need the
oracle's lse for a bounded set of tokens) and check properties that hold at
any size (bitwise shard invariance, <h, dH> = <W, dW>, zero padding rows).
"""
import numpy as np
import pytest
import torch

import workloads
from gpu_util import (assert_grad_close, assert_logp_close, dev, dev_bf16, host_bf16_to_f64)

pytestmark = pytest.mark.gpu

N_ROWS = 16       # sampled tokens checked against the oracle
N_SPARSE_G = 48   # tokens with non-zero g in the sparse-g runs
N_VROWS = 40      # sampled vocab rows of dW


@pytest.fixture(scope="module")
def rlk():
    from deterministic_token_logprob_gb300 import build
    build.build()
    import deterministic_token_logprob_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


@pytest.fixture(scope="module")
def W8b():
    w = workloads.QWEN3_8B
    bits = workloads.make_W(w.V, w.H, 0)
    return bits, dev_bf16(bits)


def _vrows(w, y, pos, seed):
    """Sampled dW rows: targets of some non-zero-g tokens (large one-hot terms),
    random rows, and padding rows at or above V_true."""
    r = list(workloads.sample_rows(w.V_true, N_VROWS - 12, seed=seed, stream=21))
    r += list(y[pos[:8]])
    r += [w.V_true, w.V - 1, w.V_true + 3, w.V - 2]
    return np.array(sorted(set(int(v) for v in r)), dtype=np.int64)


def test_qwen3_8b_forward_sampled(rlk, oracle_mod, W8b):
    w = workloads.QWEN3_8B_FWD
    bits, W = W8b
    h_bits = workloads.make_h(w.T, w.H, 0)
    y = workloads.make_y(w.T, w.V_true, 0)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    logp, lse = rlk.linear_logp_fwd(dev_bf16(h_bits), W, dev(y), w.V_true, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rows = workloads.sample_rows(w.T, N_ROWS, seed=1)
    ref_logp, ref_lse = oracle_mod.forward(h_bits, bits, y, w.V_true, rows=rows)
    assert_logp_close(logp.cpu().numpy()[rows], ref_logp)
    assert_logp_close(lse.cpu().numpy()[rows], ref_lse)
    lp = logp.cpu().numpy()
    assert np.all(np.isfinite(lp)) and np.all(lp <= 0)


def test_qwen3_8b_fwd_bwd_sampled(rlk, oracle_mod, W8b):
    w = workloads.QWEN3_8B
    bits, W = W8b
    d = workloads.make_inputs(w, with_W=False)
    g, pos = workloads.sparse_g(w.T, N_SPARSE_G, seed=2)
    h, y = dev_bf16(d["h"]), dev(d["y"])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    logp, lse = rlk.linear_logp_fwd(h, W, y, w.V_true, err_flag=err)
    dH, dW = rlk.linear_logp_bwd(h, W, y, lse, dev(g), w.V_true, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    g64 = g.astype(np.float64)
    # the oracle's lse for every token with g != 0 (the only ones dW needs)
    ref_logp_pos, ref_lse_pos = oracle_mod.forward(d["h"], bits, d["y"], w.V_true, rows=pos)
    assert_logp_close(logp.cpu().numpy()[pos], ref_logp_pos)
    lse_full = np.full(w.T, np.nan)
    lse_full[pos] = ref_lse_pos
    # dH rows: tokens with g != 0 against the oracle, tokens with g == 0 exactly zero
    rows = pos[:N_ROWS]
    ref_dH = oracle_mod.backward_dh(d["h"], bits, d["y"], g64, w.V_true, rows=rows)
    dH_h = host_bf16_to_f64(dH)
    assert_grad_close(dH_h[rows], ref_dH, what="dH rows")
    zero_rows = np.setdiff1d(workloads.sample_rows(w.T, 64, seed=3), pos)
    assert np.all(dH_h[zero_rows] == 0.0)
    vr = _vrows(w, d["y"], pos, seed=4)
    ref_dW = oracle_mod.backward_dw(d["h"], bits, d["y"], g64, lse_full, w.V_true, vrows=vr)
    dW_h = dW.cpu().numpy()
    assert_grad_close(dW_h[vr], ref_dW, what="dW rows")
    assert np.all(dW_h[w.V_true:] == 0.0)


def test_qwen3_8b_gradient_identity_dense_g(rlk, W8b):
    """<h, dH> = sum_tv dz_tv z_tv = <W, dW> for the GRPO-style dense g of the benchmark."""
    w = workloads.QWEN3_8B
    _, W = W8b
    d = workloads.make_inputs(w, with_W=False)
    h, y, g = dev_bf16(d["h"]), dev(d["y"]), dev(d["g"])
    _, lse = rlk.linear_logp_fwd(h, W, y, w.V_true)
    dH, dW = rlk.linear_logp_bwd(h, W, y, lse, g, w.V_true, dH_fp32_partial=True)
    per_row = (h.double() * dH.double()).sum(dim=1)
    a = float(per_row.sum())
    b = 0.0
    for i in range(0, w.V, 16384):
        b += float((W[i:i + 16384].double() * dW[i:i + 16384].double()).sum())
    scale = float(per_row.abs().sum())
    assert scale > 0
    assert abs(a - b) <= 1e-4 * scale, (a, b, scale)
    assert torch.all(dW[w.V_true:] == 0)


def test_qwen3_30b_tp2_sharded_sampled(rlk, oracle_mod):
    w = workloads.QWEN3_30B_TP2
    bits = workloads.make_W(w.V, w.H, 0)
    W = dev_bf16(bits)
    d = workloads.make_inputs(w, with_W=False)
    h, y = dev_bf16(d["h"]), dev(d["y"])
    assert list(w.shards) == rlk.shard_bounds(w.V, w.V_true, 2)
    logp, lse = rlk.linear_logp_fwd(h, W, y, w.V_true)
    parts = torch.stack([rlk.linear_logp_fwd(h, W[a:a + n], y, w.V_true, vocab_start=a, partial=True)
                         for a, n in w.shards])
    slogp, slse = rlk.lse_merge(parts)
    assert torch.equal(slogp, logp) and torch.equal(slse, lse)
    rows = workloads.sample_rows(w.T, N_ROWS, seed=5)
    ref_logp, _ = oracle_mod.forward(d["h"], bits, d["y"], w.V_true, rows=rows)
    assert_logp_close(slogp.cpu().numpy()[rows], ref_logp)

    g, pos = workloads.sparse_g(w.T, N_SPARSE_G, seed=6)
    gd = dev(g)
    dH_parts, dW_parts = [], []
    for a, n in w.shards:
        dHp, dWp = rlk.linear_logp_bwd(h, W[a:a + n], y, slse, gd, w.V_true, vocab_start=a,
                                       dH_fp32_partial=True)
        dH_parts.append(dHp)
        dW_parts.append(dWp)
    dH = rlk.shard_sum_bf16(torch.stack(dH_parts))
    dW = torch.cat(dW_parts)
    g64 = g.astype(np.float64)
    _, ref_lse_pos = oracle_mod.forward(d["h"], bits, d["y"], w.V_true, rows=pos)
    lse_full = np.full(w.T, np.nan)
    lse_full[pos] = ref_lse_pos
    ref_dH = oracle_mod.backward_dh(d["h"], bits, d["y"], g64, w.V_true, rows=pos[:N_ROWS])
    assert_grad_close(host_bf16_to_f64(dH)[pos[:N_ROWS]], ref_dH, what="sharded dH rows")
    vr = _vrows(w, d["y"], pos, seed=7)
    vr = np.union1d(vr, [77823, 77824])     # both sides of the shard boundary
    ref_dW = oracle_mod.backward_dw(d["h"], bits, d["y"], g64, lse_full, w.V_true, vrows=vr)
    assert_grad_close(dW.cpu().numpy()[vr], ref_dW, what="sharded dW rows")


def test_batch_invariance_full(rlk, oracle_mod, W8b):
    """128 fixed targets inside ragged batches T in {1, 7, 128, 1000, 4097} at the
    Qwen3-8B shape: bitwise identical logp, lse and dH rows across T and runs."""
    from test_gpu_determinism import _invariance
    bits, W = W8b
    w = workloads.QWEN3_8B
    _invariance(rlk, w.H, w.V, w.V_true, bits, W, workloads.INVARIANCE_T, oracle_mod)


def test_qwen3_8b_saved_logits_bitwise(rlk, W8b):
    """The saved-logits pair reproduces the recompute path bit for bit at full size."""
    w = workloads.QWEN3_8B
    _, W = W8b
    d = workloads.make_inputs(w, with_W=False)
    h, y, g = dev_bf16(d["h"]), dev(d["y"]), dev(d["g"])
    logp, lse = rlk.linear_logp_fwd(h, W, y, w.V_true)
    dH, dW = rlk.linear_logp_bwd(h, W, y, lse, g, w.V_true)
    (logp2, lse2), z = rlk.linear_logp_fwd_save(h, W, y, w.V_true)
    assert torch.equal(logp, logp2) and torch.equal(lse, lse2)
    del logp2, lse2
    dH2, dW2 = rlk.linear_logp_bwd_saved(h, W, y, lse, g, z, w.V_true)
    assert torch.equal(dH, dH2)
    assert torch.equal(dW, dW2)


def test_qwen3_8b_saved_probs_close_to_recompute(rlk, W8b):
    """The bf16 saved-probabilities pair at full size: logp / lse bitwise, dH / dW within
    the gradient tolerance of the recompute path (one extra bf16 rounding of p)."""
    from gpu_util import rel_l2
    w = workloads.QWEN3_8B
    _, W = W8b
    d = workloads.make_inputs(w, with_W=False)
    h, y, g = dev_bf16(d["h"]), dev(d["y"]), dev(d["g"])
    logp, lse = rlk.linear_logp_fwd(h, W, y, w.V_true)
    dH, dW = rlk.linear_logp_bwd(h, W, y, lse, g, w.V_true, dH_fp32_partial=True)
    (logp2, lse2), pbuf = rlk.linear_logp_fwd_save_probs(h, W, y, w.V_true)
    assert torch.equal(logp, logp2) and torch.equal(lse, lse2)
    dH2, dW2 = rlk.linear_logp_bwd_saved_probs(h, W, y, lse, g, pbuf, w.V_true, dH_fp32_partial=True)
    eH = float((dH2 - dH).norm() / dH.norm())
    eW = float((dW2 - dW).norm() / dW.norm())
    assert eH <= 1e-2 and eW <= 1e-2, (eH, eW)
    assert torch.all(dW2[w.V_true:] == 0)


def test_qwen3_30b_rank_call_sizes_batch_invariant(rlk, oracle_mod):
    # The token counts per call of the pages' own TP = 2 measurement (796, 1820, 6827) on the
    # Qwen3-30B-A3B output layer, through the two-shard path (shard statistics + merge; fp32 dH
    # partials + ordered sum). The smaller batches are prefixes of the largest, so every token
    # must get the same logp, lse and dH bits in all three calls; the merged results equal the
    # unsharded call; sampled rows match the oracle.
    w = workloads.QWEN3_30B_TP2
    bits = workloads.make_W(w.V, w.H, 0)
    W = dev_bf16(bits)
    Tmax = 6827
    hb = workloads.make_h(Tmax, w.H, 21)
    yb = workloads.make_y(Tmax, w.V_true, 21)
    g = np.random.default_rng(22).standard_normal(Tmax).astype(np.float32)
    seen = {}
    for T in (796, 1820, Tmax):
        h, y, gd = dev_bf16(hb[:T]), dev(yb[:T]), dev(g[:T])
        parts = torch.stack([rlk.linear_logp_fwd(h, W[a:a + n], y, w.V_true, vocab_start=a,
                                                 partial=True) for a, n in w.shards])
        logp, lse = rlk.lse_merge(parts)
        ulogp, ulse = rlk.linear_logp_fwd(h, W, y, w.V_true)
        assert torch.equal(logp, ulogp) and torch.equal(lse, ulse), T
        dHp = torch.stack([rlk.linear_logp_bwd(h, W[a:a + n], y, lse, gd, w.V_true, vocab_start=a,
                                               dH_fp32_partial=True, want_dW=False)[0]
                           for a, n in w.shards])
        dH = rlk.shard_sum_bf16(dHp)
        seen[T] = (logp.cpu().numpy(), lse.cpu().numpy(), dH.view(torch.int16).cpu().numpy())
    for T in (796, 1820):
        for i, what in enumerate(("logp", "lse", "dH")):   # compared as raw bits
            assert np.array_equal(seen[T][i].view(np.int32 if i < 2 else np.int16),
                                  seen[Tmax][i][:T].view(np.int32 if i < 2 else np.int16)), (T, what)
    rows = workloads.sample_rows(796, 16, seed=23)
    ref_logp, _ = oracle_mod.forward(hb[:796], bits, yb[:796], w.V_true, rows=rows)
    assert_logp_close(seen[796][0][rows], ref_logp)
    ref_dH = oracle_mod.backward_dh(hb[:796], bits, yb[:796], g[:796].astype(np.float64), w.V_true,
                                    rows=rows[:8])
    dH_bits = seen[796][2][rows[:8]].view(np.uint16).astype(np.uint32) << 16   # bf16 -> fp32 bits
    assert_grad_close(dH_bits.view(np.float32).astype(np.float64), ref_dH, what="dH rows")
