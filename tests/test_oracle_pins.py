"""Pins for the fp64 oracle, each against something other than the oracle itself.

Every oracle function is checked against at least one of: a hand-derived
worked example, a closed form, an invariant of the mathematics, a textbook
special case evaluated with Python's ``math``, central finite differences, or
a brute-force evaluation by a different tool (numpy) on tiny inputs. The set is
chosen so that a dropped term, a wrong sign, a wrong index or a transposed
operand in the oracle fails at least one test.
"""
import math
import os

import numpy as np
import pytest

import workloads

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                vals[k] = float(v)
    return vals


def _rand(rng, T, H, V, scale=1.0):
    h = rng.standard_normal((T, H)) * scale
    W = rng.standard_normal((V, H)) * scale
    return h, W


# --------------------------------------------------------------------------- bf16


def test_bf16_widening_known_bit_patterns(oracle_mod):
    cases = {0x3F80: 1.0, 0xC000: -2.0, 0x3F00: 0.5, 0x3F81: 1.0078125, 0x4049: 3.140625,
             0x0000: 0.0, 0x0001: 2.0 ** -133, 0x7F7F: 3.3895313892515355e38}
    for bits, val in cases.items():
        assert oracle_mod.bf16_to_double(bits) == val, hex(bits)
    assert math.isinf(oracle_mod.bf16_to_double(0x7F80))
    assert math.copysign(1.0, oracle_mod.bf16_to_double(0x8000)) == -1.0


def test_bf16_mode_equals_f64_mode_on_widened_values(oracle_mod):
    rng = np.random.default_rng(1)
    hb = workloads.bf16_bits(rng.standard_normal((5, 24)).astype(np.float32))
    Wb = workloads.bf16_bits((rng.standard_normal((40, 24)) * 0.3).astype(np.float32))
    y = rng.integers(0, 33, 5)
    h64 = workloads.bf16_to_f32(hb).astype(np.float64)
    W64 = workloads.bf16_to_f32(Wb).astype(np.float64)
    a = oracle_mod.forward(hb, Wb, y, 33)
    b = oracle_mod.forward(h64, W64, y, 33)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
    g = rng.standard_normal(5)
    np.testing.assert_array_equal(oracle_mod.backward_dh(hb, Wb, y, g, 33),
                                  oracle_mod.backward_dh(h64, W64, y, g, 33))
    np.testing.assert_array_equal(oracle_mod.backward_dw(hb, Wb, y, g, a[1], 33),
                                  oracle_mod.backward_dw(h64, W64, y, g, b[1], 33))


# --------------------------------------------------------------------------- forward


def test_worked_example_forward(oracle_mod):
    gold = _golden("worked_example_3class.txt")
    h = np.array([[1.0, 0.0]] * 3)
    W = np.array([[1.0, 0.0], [0.0, 1.0], [-1.0, 0.0], [7.0, 7.0]])
    logp, lse = oracle_mod.forward(h, W, np.array([0, 1, 2]), V_true=3)
    np.testing.assert_allclose(lse, gold["lse"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(logp, [gold["logp_y0"], gold["logp_y1"], gold["logp_y2"]], rtol=0, atol=1e-14)


def test_worked_example_backward(oracle_mod):
    gold = _golden("worked_example_3class.txt")
    h = np.array([[1.0, 0.0]])
    W = np.array([[1.0, 0.0], [0.0, 1.0], [-1.0, 0.0], [7.0, 7.0]])
    y = np.array([0])
    g = np.array([2.0])
    dH = oracle_mod.backward_dh(h, W, y, g, V_true=3)
    np.testing.assert_allclose(dH[0], [gold["dH_0"], gold["dH_1"]], rtol=0, atol=1e-14)
    _, lse = oracle_mod.forward(h, W, y, 3)
    dW = oracle_mod.backward_dw(h, W, y, g, lse, V_true=3)
    exp = np.array([[gold["dW_00"], 0], [gold["dW_10"], 0], [gold["dW_20"], 0], [0, 0]])
    np.testing.assert_allclose(dW, exp, rtol=0, atol=1e-14)


def test_zero_weights_give_minus_log_vtrue(oracle_mod):
    rng = np.random.default_rng(2)
    T, H, V, Vt = 6, 16, 50, 37
    h = rng.standard_normal((T, H))
    W = np.zeros((V, H))
    W[Vt:] = rng.standard_normal((V - Vt, H)) * 5   # padding rows must not count
    logp, lse = oracle_mod.forward(h, W, rng.integers(0, Vt, T), Vt)
    np.testing.assert_allclose(logp, -math.log(Vt), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, math.log(Vt), rtol=0, atol=1e-13)


def test_identical_weight_rows_give_minus_log_vtrue(oracle_mod):
    rng = np.random.default_rng(3)
    T, H, V = 4, 9, 21
    h = rng.standard_normal((T, H))
    W = np.tile(rng.standard_normal(H), (V, 1))
    logp, _ = oracle_mod.forward(h, W, rng.integers(0, V, T), V)
    np.testing.assert_allclose(logp, -math.log(V), rtol=0, atol=1e-12)


def test_single_class_gives_zero_logp_and_zero_grad(oracle_mod):
    rng = np.random.default_rng(4)
    h, W = _rand(rng, 3, 7, 5)
    y = np.zeros(3, np.int64)
    g = rng.standard_normal(3)
    logp, lse = oracle_mod.forward(h, W, y, V_true=1)
    np.testing.assert_allclose(logp, 0.0, atol=1e-15)
    np.testing.assert_allclose(lse, h @ W[0], rtol=1e-13)
    assert np.all(oracle_mod.backward_dh(h, W, y, g, 1) == 0.0)
    assert np.all(oracle_mod.backward_dw(h, W, y, g, lse, 1) == 0.0)


def test_two_classes_match_logistic_closed_form(oracle_mod):
    # logp(y) = -log(1 + exp(z_other - z_y)) = -softplus(z_other - z_y)
    rng = np.random.default_rng(5)
    h, W = _rand(rng, 8, 3, 2)
    y = rng.integers(0, 2, 8)
    logp, _ = oracle_mod.forward(h, W, y, 2)
    for t in range(8):
        zy = sum(h[t, k] * W[y[t], k] for k in range(3))
        zo = sum(h[t, k] * W[1 - y[t], k] for k in range(3))
        assert logp[t] == pytest.approx(-math.log1p(math.exp(zo - zy)), abs=1e-14)


def test_softmax_over_all_targets_sums_to_one(oracle_mod):
    rng = np.random.default_rng(6)
    T, H, V, Vt = 3, 11, 40, 29
    h, W = _rand(rng, T, H, V, 0.7)
    for t in range(T):
        hs = np.repeat(h[t:t + 1], Vt, axis=0)
        logp, _ = oracle_mod.forward(hs, W, np.arange(Vt), Vt)
        assert math.fsum(math.exp(x) for x in logp) == pytest.approx(1.0, abs=1e-14)
        assert np.all(logp <= 0.0)


def test_brute_force_numpy_small(oracle_mod):
    rng = np.random.default_rng(7)
    T, H, V, Vt = 13, 32, 70, 61
    h, W = _rand(rng, T, H, V, 0.5)
    y = rng.integers(0, Vt, T)
    z = (h @ W.T)[:, :Vt]
    lse_ref = np.logaddexp.reduce(z, axis=1)
    logp_ref = z[np.arange(T), y] - lse_ref
    logp, lse = oracle_mod.forward(h, W, y, Vt)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(logp, logp_ref, rtol=1e-13, atol=1e-13)


def test_large_logits_are_max_shifted(oracle_mod):
    h = np.array([[1.0], [1.0], [1.0]])
    W = np.array([[1000.0], [0.0], [-1000.0]])
    logp, lse = oracle_mod.forward(h, W, np.array([0, 1, 2]), 3)
    assert lse[0] == pytest.approx(1000.0, abs=1e-12)
    assert logp[0] == pytest.approx(0.0, abs=1e-12)
    assert logp[1] == pytest.approx(-1000.0, abs=1e-12)
    assert logp[2] == pytest.approx(-2000.0, abs=1e-9)


def test_padding_rows_have_no_effect(oracle_mod):
    rng = np.random.default_rng(8)
    T, H, V, Vt = 5, 12, 30, 22
    h, W = _rand(rng, T, H, V)
    y = rng.integers(0, Vt, T)
    g = rng.standard_normal(T)
    a = oracle_mod.forward(h, W, y, Vt)
    W2 = W.copy()
    W2[Vt:] = rng.standard_normal((V - Vt, H)) * 100
    b = oracle_mod.forward(h, W2, y, Vt)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(oracle_mod.backward_dh(h, W, y, g, Vt),
                                  oracle_mod.backward_dh(h, W2, y, g, Vt))
    dW = oracle_mod.backward_dw(h, W, y, g, a[1], Vt)
    assert np.all(dW[Vt:] == 0.0)


def test_shift_invariance(oracle_mod):
    # adding c to every weight row adds h.c to every logit of the token: logp unchanged
    rng = np.random.default_rng(9)
    T, H, V = 6, 10, 25
    h, W = _rand(rng, T, H, V)
    y = rng.integers(0, V, T)
    c = rng.standard_normal(H) * 3
    a, la = oracle_mod.forward(h, W, y, V)
    b, lb = oracle_mod.forward(h, W + c, y, V)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lb - la, h @ c, rtol=0, atol=1e-12)


def test_row_subset_matches_full(oracle_mod):
    rng = np.random.default_rng(10)
    T, H, V = 17, 8, 19
    h, W = _rand(rng, T, H, V)
    y = rng.integers(0, V, T)
    g = rng.standard_normal(T)
    rows = np.array([16, 0, 5, 5, 9])
    full = oracle_mod.forward(h, W, y, V)
    sub = oracle_mod.forward(h, W, y, V, rows=rows)
    np.testing.assert_array_equal(sub[0], full[0][rows])
    dh_full = oracle_mod.backward_dh(h, W, y, g, V)
    np.testing.assert_array_equal(oracle_mod.backward_dh(h, W, y, g, V, rows=rows), dh_full[rows])
    dw_full = oracle_mod.backward_dw(h, W, y, g, full[1], V)
    vr = np.array([3, 18, 0])
    np.testing.assert_array_equal(oracle_mod.backward_dw(h, W, y, g, full[1], V, vrows=vr), dw_full[vr])


def test_invalid_targets(oracle_mod):
    rng = np.random.default_rng(11)
    T, H, V, Vt = 4, 6, 12, 9
    h, W = _rand(rng, T, H, V)
    y = np.array([3, -1, 9, 8])   # -1 and 9 (>= V_true) are invalid
    g = np.ones(T)
    logp, lse = oracle_mod.forward(h, W, y, Vt)
    assert np.isnan(logp[1]) and np.isnan(logp[2])
    assert np.isfinite(logp[0]) and np.isfinite(logp[3])
    dH = oracle_mod.backward_dh(h, W, y, g, Vt)
    assert np.all(dH[1] == 0) and np.all(dH[2] == 0)
    keep = np.array([1.0, 0.0, 0.0, 1.0])
    dW_a = oracle_mod.backward_dw(h, W, y, g, lse, Vt)
    dW_b = oracle_mod.backward_dw(h, W, y, keep, lse, Vt)
    np.testing.assert_array_equal(dW_a, dW_b)


# --------------------------------------------------------------------------- backward


def _loss(oracle_mod, h, W, y, g, Vt):
    logp, _ = oracle_mod.forward(h, W, y, Vt)
    return float(np.dot(g, logp))


def test_finite_differences(oracle_mod):
    rng = np.random.default_rng(12)
    T, H, V, Vt = 3, 5, 7, 6
    h, W = _rand(rng, T, H, V, 0.8)
    y = np.array([0, 5, 2])
    g = rng.standard_normal(T)
    dH = oracle_mod.backward_dh(h, W, y, g, Vt)
    _, lse = oracle_mod.forward(h, W, y, Vt)
    dW = oracle_mod.backward_dw(h, W, y, g, lse, Vt)
    eps = 1e-6
    fd_h = np.zeros_like(h)
    for t in range(T):
        for k in range(H):
            hp, hm = h.copy(), h.copy()
            hp[t, k] += eps
            hm[t, k] -= eps
            fd_h[t, k] = (_loss(oracle_mod, hp, W, y, g, Vt) - _loss(oracle_mod, hm, W, y, g, Vt)) / (2 * eps)
    fd_w = np.zeros_like(W)
    for v in range(V):
        for k in range(H):
            Wp, Wm = W.copy(), W.copy()
            Wp[v, k] += eps
            Wm[v, k] -= eps
            fd_w[v, k] = (_loss(oracle_mod, h, Wp, y, g, Vt) - _loss(oracle_mod, h, Wm, y, g, Vt)) / (2 * eps)
    assert np.linalg.norm(dH - fd_h) <= 1e-6 * np.linalg.norm(fd_h)
    assert np.linalg.norm(dW - fd_w) <= 1e-6 * np.linalg.norm(fd_w)
    assert np.all(fd_w[Vt:] == 0.0) and np.all(dW[Vt:] == 0.0)


def test_gradient_invariants(oracle_mod):
    # sum_v dz[t][v] = 0  =>  sum_v dW_v = 0 ; and <h, dH> = <W, dW> = sum dz * z
    rng = np.random.default_rng(13)
    T, H, V, Vt = 9, 14, 33, 30
    h, W = _rand(rng, T, H, V, 0.6)
    y = rng.integers(0, Vt, T)
    g = rng.standard_normal(T)
    _, lse = oracle_mod.forward(h, W, y, Vt)
    dH = oracle_mod.backward_dh(h, W, y, g, Vt)
    dW = oracle_mod.backward_dw(h, W, y, g, lse, Vt)
    scale = np.abs(dW).sum()
    np.testing.assert_allclose(dW.sum(axis=0), 0.0, atol=1e-13 * scale)
    a = float(np.sum(h * dH))
    b = float(np.sum(W * dW))
    assert a == pytest.approx(b, rel=1e-12, abs=1e-12)


def test_sparse_g_skips_exactly(oracle_mod):
    rng = np.random.default_rng(14)
    T, H, V = 12, 6, 15
    h, W = _rand(rng, T, H, V)
    y = rng.integers(0, V, T)
    g = np.zeros(T)
    g[[2, 7]] = [0.5, -1.5]
    _, lse = oracle_mod.forward(h, W, y, V)
    lse_masked = np.full(T, np.nan)
    lse_masked[[2, 7]] = lse[[2, 7]]
    np.testing.assert_array_equal(oracle_mod.backward_dw(h, W, y, g, lse, V),
                                  oracle_mod.backward_dw(h, W, y, g, lse_masked, V))


# --------------------------------------------------------------------------- shards


@pytest.mark.parametrize("splits", [[0, 40], [0, 17, 40], [0, 8, 16, 24, 40], [0, 35, 40]])
def test_shard_stats_merge_equals_full(oracle_mod, splits):
    rng = np.random.default_rng(15)
    T, H, V, Vt = 7, 9, 40, 33
    h, W = _rand(rng, T, H, V)
    y = rng.integers(0, Vt, T)
    y[0] = 0
    y[1] = Vt - 1
    full_logp, full_lse = oracle_mod.forward(h, W, y, Vt)
    parts = [oracle_mod.shard_stats(h, W[a:b], y, a, Vt) for a, b in zip(splits[:-1], splits[1:])]
    m = np.stack([p[0] for p in parts])
    s = np.stack([p[1] for p in parts])
    zt = np.stack([p[2] for p in parts])
    logp, lse = oracle_mod.lse_merge(m, s, zt)
    np.testing.assert_allclose(lse, full_lse, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(logp, full_logp, rtol=1e-13, atol=1e-13)
    # exactly one shard owns each target
    assert np.all(np.isfinite(zt).sum(axis=0) == 1)


def test_shard_stats_brute_force(oracle_mod):
    rng = np.random.default_rng(16)
    T, H, Vl, start, Vt = 4, 5, 10, 20, 26   # columns 20..29, of which 20..25 are valid
    h = rng.standard_normal((T, H))
    Wl = rng.standard_normal((Vl, H))
    y = np.array([21, 3, 25, 26])
    m, s, zt = oracle_mod.shard_stats(h, Wl, y, start, Vt)
    z = h @ Wl[:Vt - start].T
    np.testing.assert_allclose(m, z.max(axis=1), rtol=1e-14)
    np.testing.assert_allclose(s, np.exp(z - z.max(axis=1, keepdims=True)).sum(axis=1), rtol=1e-13)
    assert zt[0] == pytest.approx(z[0, 1], rel=1e-14)
    assert zt[1] == -math.inf
    assert zt[2] == pytest.approx(z[2, 5], rel=1e-14)
    assert math.isnan(zt[3])   # 26 >= V_true: invalid target
    # a shard entirely above V_true is empty
    m, s, zt = oracle_mod.shard_stats(h, Wl, np.array([1, 2, 3, 4]), 40, 30)
    assert np.all(m == -math.inf) and np.all(s == 0.0) and np.all(zt == -math.inf)


def test_lse_merge_brute_force(oracle_mod):
    rng = np.random.default_rng(17)
    S, T = 5, 11
    m = rng.standard_normal((S, T)) * 20
    s = rng.uniform(1.0, 1e4, (S, T))
    zt = np.full((S, T), -math.inf)
    owner = rng.integers(0, S, T)
    zt[owner, np.arange(T)] = rng.standard_normal(T) * 5
    s[2, 3] = 0.0
    m[2, 3] = -math.inf     # an empty shard for token 3
    logp, lse = oracle_mod.lse_merge(m, s, zt)
    for t in range(T):
        ref = math.log(math.fsum(s[i, t] * math.exp(m[i, t]) for i in range(S) if s[i, t] > 0))
        assert lse[t] == pytest.approx(ref, rel=1e-13, abs=1e-12)
        assert logp[t] == pytest.approx(zt[owner[t], t] - ref, rel=1e-13, abs=1e-12)
    # S = 1: lse = m + log s
    l1, s1 = oracle_mod.lse_merge(m[:1], s[:1], zt[:1])
    np.testing.assert_allclose(s1, m[0] + np.log(s[0]), rtol=1e-15)
    # a NaN target anywhere propagates
    zt[1, 4] = math.nan
    logp, _ = oracle_mod.lse_merge(m, s, zt)
    assert math.isnan(logp[4])
