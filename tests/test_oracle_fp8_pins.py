"""Pins for the oracle's FP8 (E4M3, one power-of-two scale per row) LM-head pieces.

Each check compares the oracle with something other than itself: PyTorch's
float8_e4m3fn conversions (a library routine for the format and its
round-to-nearest-even), values of the format fixed by its definition, the two
inequalities that define the row scale, the half-spacing error bound, and
closed forms of the straight-through backward when every logit is equal
(uniform softmax). A wrong exponent bias, a dropped subnormal, ties rounded
away from even, a scale one power of two off, or a straight-through gradient
contracted with the quantized instead of the unquantized operand fails one of
them.
"""
import math

import numpy as np
import pytest
import torch

import workloads

E4M3_MAX = 448.0


def _torch_decode_all():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _torch_codes(y):
    """E4M3 codes of float values |y| <= 448 by PyTorch's float -> float8_e4m3fn cast."""
    t = torch.from_numpy(np.ascontiguousarray(y, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def _deq(q, s):
    return _torch_decode_all()[q] * s[:, None]


# --------------------------------------------------------------------------- format


def test_e4m3_decode_matches_torch_for_every_code(oracle_mod):
    ref = _torch_decode_all()
    for c in range(256):
        v = oracle_mod.e4m3_to_double(c)
        if math.isnan(ref[c]):
            assert math.isnan(v), hex(c)
        else:
            assert v == ref[c] and math.copysign(1, v) == math.copysign(1, ref[c]), hex(c)


def test_e4m3_known_values(oracle_mod):
    known = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
             0x39: 1.125, 0x40: 2.0, 0x77: 240.0, 0x7E: 448.0, 0xB8: -1.0, 0xFE: -448.0}
    for c, v in known.items():
        assert oracle_mod.e4m3_to_double(c) == v, hex(c)
    assert math.isnan(oracle_mod.e4m3_to_double(0x7F)) and math.isnan(oracle_mod.e4m3_to_double(0xFF))
    # positive codes 0..126 are strictly increasing (the rounding search relies on it)
    vals = [oracle_mod.e4m3_to_double(c) for c in range(127)]
    assert all(a < b for a, b in zip(vals, vals[1:]))


# --------------------------------------------------------------------------- quantizer


def _scale_is_minimal(x, s):
    amax = np.abs(x).max(axis=1)
    for a, sc in zip(amax, s):
        e = math.log2(sc)
        assert e == int(e), sc
        if a == 0:
            assert sc == 1.0
        else:
            assert a <= E4M3_MAX * sc, (a, sc)
            assert a > E4M3_MAX * sc / 2, (a, sc)


def test_quantize_scale_definition_and_codes_match_torch(oracle_mod):
    rng = np.random.default_rng(7)
    x = rng.standard_normal((12, 96)) * np.exp2(rng.integers(-20, 20, 12))[:, None]
    x[3] = 0.0                                       # all-zero row -> scale 1, codes 0
    x[4, 5] = 448.0 * 2.0 ** 3                       # amax exactly 448 * 2^e -> e = 3
    x[5, 0] = 448.0 * 2.0 ** -2 * (1 + 2.0 ** -40)   # just above -> the next power
    bits = workloads.bf16_bits(x.astype(np.float32))
    xb = workloads.bf16_to_f32(bits).astype(np.float64)
    for inp, xv in ((x, x), (bits, xb)):
        q, s = oracle_mod.quantize_rows_e4m3(inp)
        _scale_is_minimal(xv, s)
        assert np.all(q[3] == 0) and s[3] == 1.0
        np.testing.assert_array_equal(q, _torch_codes(xv / s[:, None]))
    q, s = oracle_mod.quantize_rows_e4m3(x)
    assert s[4] == 8.0 and s[5] == 2.0 ** -1


def test_quantize_ties_to_even(oracle_mod):
    vals = np.array([oracle_mod.e4m3_to_double(c) for c in range(127)])
    mids = (vals[:-1] + vals[1:]) / 2                 # exact midpoints between neighbours
    row = np.concatenate([[E4M3_MAX], mids, -mids])[None, :]   # amax 448 -> scale 1
    q, s = oracle_mod.quantize_rows_e4m3(row)
    assert s[0] == 1.0
    n = len(mids)
    lo = np.arange(n)
    expect = np.where(lo % 2 == 0, lo, lo + 1)        # the even code of each pair
    np.testing.assert_array_equal(q[0, 1:1 + n], expect)
    np.testing.assert_array_equal(q[0, 1 + n:], expect | 0x80)
    np.testing.assert_array_equal(q, _torch_codes(row))


def test_quantize_error_within_half_spacing(oracle_mod):
    rng = np.random.default_rng(8)
    x = rng.standard_normal((8, 256)) * 0.02
    q, s = oracle_mod.quantize_rows_e4m3(x)
    deq = _deq(q, s)
    y = np.abs(x) / s[:, None]
    # spacing of E4M3 around y: 2^(floor(log2 y) - 3) for normals (y >= 2^-6), 2^-9 below
    expo = np.floor(np.log2(np.maximum(y, 2.0 ** -6)))
    half = np.exp2(expo - 3) / 2 * s[:, None]
    assert np.all(np.abs(x - deq) <= half * (1 + 1e-12))
    # odd symmetry
    qn, sn = oracle_mod.quantize_rows_e4m3(-x)
    assert np.array_equal(sn, s)
    nz = q != 0
    np.testing.assert_array_equal(qn[nz], q[nz] ^ 0x80)


# --------------------------------------------------------------------------- fp8 forward / STE backward


def test_e4m3_operands_equal_their_decoded_values(oracle_mod):
    """The oracle's E4M3 operand path equals its float64 path on values decoded by PyTorch."""
    rng = np.random.default_rng(9)
    T, H, V, Vt = 6, 48, 70, 64
    h = rng.standard_normal((T, H))
    W = rng.standard_normal((V, H)) * 0.05
    y = rng.integers(0, Vt, T)
    hq, Wq = oracle_mod.quantize_rows_e4m3(h), oracle_mod.quantize_rows_e4m3(W)
    a = oracle_mod.forward(hq, Wq, y, Vt)
    b = oracle_mod.forward(_deq(*hq), _deq(*Wq), y, Vt)
    np.testing.assert_allclose(a[0], b[0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(a[1], b[1], rtol=0, atol=1e-12)
    m, s_, zt = oracle_mod.shard_stats(hq, (Wq[0][32:], Wq[1][32:]), y, 32, Vt)
    m2, s2, zt2 = oracle_mod.shard_stats(_deq(*hq), _deq(*Wq)[32:], y, 32, Vt)
    np.testing.assert_allclose(np.stack([m, s_]), np.stack([m2, s2]), rtol=1e-12)
    np.testing.assert_array_equal(np.isinf(zt), np.isinf(zt2))


def test_ste_uniform_softmax_closed_forms(oracle_mod):
    """Zero logit operands make p uniform over V_true: dH_t = g_t (W_{y_t} - mean_v W_v),
    dW_v = sum_t g_t (1[v = y_t] - 1/V_true) h_t, with the UNquantized h and W."""
    rng = np.random.default_rng(10)
    T, H, V, Vt = 5, 32, 40, 36
    h = rng.standard_normal((T, H))
    W = rng.standard_normal((V, H))
    y = rng.integers(0, Vt, T)
    g = rng.standard_normal(T)
    zero_W = (np.zeros((V, H), np.uint8), np.ones(V))
    hq = oracle_mod.quantize_rows_e4m3(h)
    dH = oracle_mod.backward_dh_ste(hq, zero_W, h, W, y, g, Vt)
    ref = g[:, None] * (W[y] - W[:Vt].mean(axis=0))
    np.testing.assert_allclose(dH, ref, rtol=1e-12, atol=1e-12)
    lse = np.full(T, math.log(Vt))
    dW = oracle_mod.backward_dw_ste(hq, zero_W, h, y, g, lse, Vt)
    onehot = np.zeros((T, V))
    onehot[np.arange(T), y] = 1.0
    refW = (onehot[:, :Vt] - 1.0 / Vt).T @ (g[:, None] * h)
    np.testing.assert_allclose(dW[:Vt], refW, rtol=1e-12, atol=1e-12)
    assert np.all(dW[Vt:] == 0)
    # zero h operand for the logits: the same uniform softmax
    zero_h = (np.zeros((T, H), np.uint8), np.ones(T))
    Wq = oracle_mod.quantize_rows_e4m3(W)
    np.testing.assert_allclose(oracle_mod.backward_dh_ste(zero_h, Wq, h, W, y, g, Vt), ref,
                               rtol=1e-12, atol=1e-12)


def test_ste_equals_plain_backward_when_quantization_is_exact(oracle_mod):
    """Operands whose values are already E4M3 values times the row scale quantize to
    themselves, so the straight-through gradient is the plain gradient."""
    rng = np.random.default_rng(11)
    T, H, V, Vt = 4, 24, 30, 30
    dec = _torch_decode_all()
    grid = dec[rng.integers(0, 127, (T + V, H))] * np.where(rng.random((T + V, H)) < 0.5, -1, 1)
    grid[:, 0] = 448.0                                   # every row's scale is 1
    h, W = grid[:T] * 2.0 ** -8, grid[T:] * 2.0 ** -12    # power-of-two row scales
    y = rng.integers(0, Vt, T)
    g = rng.standard_normal(T)
    hq, Wq = oracle_mod.quantize_rows_e4m3(h), oracle_mod.quantize_rows_e4m3(W)
    np.testing.assert_array_equal(_deq(*hq), h)
    np.testing.assert_array_equal(_deq(*Wq), W)
    a = oracle_mod.backward_dh_ste(hq, Wq, h, W, y, g, Vt)
    b = oracle_mod.backward_dh(h, W, y, g, Vt)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-15)
    _, lse = oracle_mod.forward(h, W, y, Vt)
    a = oracle_mod.backward_dw_ste(hq, Wq, h, y, g, lse, Vt)
    b = oracle_mod.backward_dw(h, W, y, g, lse, Vt)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-15)


def test_quantizer_rejects_non_finite(oracle_mod):
    x = np.ones((2, 4))
    x[1, 2] = np.inf
    with pytest.raises(RuntimeError):
        oracle_mod.quantize_rows_e4m3(x)
