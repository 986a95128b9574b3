"""fp64 CPU oracle for `linear_logp` -- TEST INFRASTRUCTURE.

Only the test-suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. The product library never does, and this package
shares no code with it: the arithmetic lives in ``rlk_oracle.c`` (plain C99,
binary64), compiled by :func:`build` with gcc.

Inputs ``h`` and ``W`` are numpy arrays either of dtype float64 or of dtype
uint16 holding raw bf16 bit patterns (the exact values the GPU receives), or
E4M3-quantized operands given as a pair ``(codes, scale)``: uint8 codes
[rows, H] and one float64 scale per row, the value of an element being
decode(code) * scale (see :func:`quantize_rows_e4m3`). Each function states the
definition it evaluates; the C file cites the passages.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rlk_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "librlk_oracle.so")

F64 = 0
BF16 = 1
E4M3 = 2


class _E4M3Rows(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scale", ctypes.c_void_p)]

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile rlk_oracle.c into oracle/_build/librlk_oracle.so (no fast-math, no FP contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=gnu99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-pthread", "-Wall", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            I = ctypes.c_int
            lib.rlko_forward.argtypes = [I, P, P, P, I64, I64, I64, I64, P, I64, P, P, I]
            lib.rlko_shard_stats.argtypes = [I, P, P, P, I64, I64, I64, I64, I64, P, I64, P, P, P, I]
            lib.rlko_lse_merge.argtypes = [P, P, P, I64, I64, P, P]
            lib.rlko_backward_dh.argtypes = [I, P, P, P, P, I64, I64, I64, I64, P, I64, P, I]
            lib.rlko_backward_dw.argtypes = [I, P, P, P, P, P, I64, I64, I64, I64, P, I64, P, I]
            lib.rlko_backward_dh_ste.argtypes = [I, P, P, I, P, P, P, P, I64, I64, I64, I64, P,
                                                 I64, P, I]
            lib.rlko_backward_dw_ste.argtypes = [I, P, P, I, P, P, P, P, I64, I64, I64, I64, P,
                                                 I64, P, I]
            lib.rlko_quantize_rows_e4m3.argtypes = [I, P, I64, I64, P, P, I]
            lib.rlko_e4m3_to_double.argtypes = [ctypes.c_uint8]
            lib.rlko_e4m3_to_double.restype = ctypes.c_double
            lib.rlko_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.rlko_bf16_to_double.restype = ctypes.c_double
            lib.rlko_default_threads.argtypes = []
            for name in ("rlko_forward", "rlko_shard_stats", "rlko_lse_merge",
                         "rlko_backward_dh", "rlko_backward_dw", "rlko_default_threads",
                         "rlko_backward_dh_ste", "rlko_backward_dw_ste", "rlko_quantize_rows_e4m3"):
                getattr(lib, name).restype = ctypes.c_int
            _lib = lib
    return _lib


def default_threads() -> int:
    """Number of host threads the oracle uses when nthreads=0 (all online cores)."""
    return int(_load().rlko_default_threads())


def bf16_to_double(bits: int) -> float:
    return float(_load().rlko_bf16_to_double(int(bits) & 0xFFFF))


class _Operand:
    """One matrix operand as the C side takes it: a kind code, a pointer, a shape.
    Keeps the arrays (and, for E4M3, the descriptor struct) alive."""

    def __init__(self, a):
        if isinstance(a, tuple):
            codes, scale = a
            codes = np.ascontiguousarray(codes)
            scale = np.ascontiguousarray(scale, dtype=np.float64)
            if codes.dtype != np.uint8 or codes.ndim != 2 or scale.shape != (codes.shape[0],):
                raise TypeError("E4M3 operands are (uint8 codes [rows, H], float64 scale [rows])")
            self.kind, self.shape, self._keep = E4M3, codes.shape, (codes, scale)
            self._desc = _E4M3Rows(codes.ctypes.data, scale.ctypes.data)
            self.ptr = ctypes.cast(ctypes.pointer(self._desc), ctypes.c_void_p)
            return
        if a.dtype == np.float64:
            self.kind = F64
        elif a.dtype == np.uint16:
            self.kind = BF16
        else:
            raise TypeError(f"oracle inputs must be float64, uint16 (bf16 bits) or (codes, scale), got {a.dtype}")
        a = np.ascontiguousarray(a)
        if a.ndim != 2:
            raise ValueError("operands are 2-D")
        self.shape, self._keep, self.ptr = a.shape, a, a.ctypes.data_as(ctypes.c_void_p)


def _pair(h, W):
    oh, ow = _Operand(h), _Operand(W)
    if oh.kind != ow.kind:
        raise TypeError("h and W must have the same element kind")
    if oh.shape[1] != ow.shape[1]:
        raise ValueError(f"shape mismatch h{oh.shape} W{ow.shape}")
    return oh.kind, oh, ow


def _ptr(a):
    if a is None:
        return None
    if isinstance(a, _Operand):
        return a.ptr
    return a.ctypes.data_as(ctypes.c_void_p)


def _rows(rows, T):
    if rows is None:
        return None, T
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    return r, int(r.shape[0])


def _check(rc, name):
    if rc != 0:
        raise RuntimeError(f"{name} failed with code {rc}")


def forward(h, W, y, V_true, rows=None, nthreads=0):
    """logp[i] = z[t][y_t] - logsumexp_{v<V_true} z[t][v], lse[i], for t = rows[i] (all tokens if None)."""
    kind, h, W = _pair(h, W)
    y = np.ascontiguousarray(y, dtype=np.int64)
    T, H = h.shape
    V = W.shape[0]
    r, n = _rows(rows, T)
    logp = np.empty(n, np.float64)
    lse = np.empty(n, np.float64)
    _check(_load().rlko_forward(kind, _ptr(h), _ptr(W), _ptr(y), T, H, V, int(V_true), _ptr(r), n,
                                _ptr(logp), _ptr(lse), int(nthreads)), "rlko_forward")
    return logp, lse


def shard_stats(h, W_local, y, vocab_start, V_true, rows=None, nthreads=0):
    """Per-token (m, s, zt) of one vocab shard holding global columns [vocab_start, vocab_start+V_local)."""
    kind, h, W_local = _pair(h, W_local)
    y = np.ascontiguousarray(y, dtype=np.int64)
    T, H = h.shape
    V_local = W_local.shape[0]
    r, n = _rows(rows, T)
    m = np.empty(n, np.float64)
    s = np.empty(n, np.float64)
    zt = np.empty(n, np.float64)
    _check(_load().rlko_shard_stats(kind, _ptr(h), _ptr(W_local), _ptr(y), T, H, V_local,
                                    int(vocab_start), int(V_true), _ptr(r), n, _ptr(m), _ptr(s),
                                    _ptr(zt), int(nthreads)), "rlko_shard_stats")
    return m, s, zt


def lse_merge(m, s, zt):
    """Merge [S, T] shard triples: lse = log sum_i s_i e^{m_i}; logp = zt_owner - lse."""
    m = np.ascontiguousarray(m, dtype=np.float64)
    s = np.ascontiguousarray(s, dtype=np.float64)
    zt = np.ascontiguousarray(zt, dtype=np.float64)
    if m.ndim != 2 or m.shape != s.shape or m.shape != zt.shape:
        raise ValueError("m, s, zt must share one [S, T] shape")
    S, T = m.shape
    logp = np.empty(T, np.float64)
    lse = np.empty(T, np.float64)
    _check(_load().rlko_lse_merge(_ptr(m), _ptr(s), _ptr(zt), S, T, _ptr(logp), _ptr(lse)),
           "rlko_lse_merge")
    return logp, lse


def backward_dh(h, W, y, g, V_true, rows=None, nthreads=0):
    """dH rows (for t = rows[i]) of L = sum_t g_t logp_t: dH_t = sum_v g_t (1[v=y_t] - p_tv) W_v."""
    kind, h, W = _pair(h, W)
    y = np.ascontiguousarray(y, dtype=np.int64)
    g = np.ascontiguousarray(g, dtype=np.float64)
    T, H = h.shape
    V = W.shape[0]
    r, n = _rows(rows, T)
    dH = np.empty((n, H), np.float64)
    _check(_load().rlko_backward_dh(kind, _ptr(h), _ptr(W), _ptr(y), _ptr(g), T, H, V, int(V_true),
                                    _ptr(r), n, _ptr(dH), int(nthreads)), "rlko_backward_dh")
    return dH


def backward_dw(h, W, y, g, lse, V_true, vrows=None, nthreads=0):
    """dW rows (for v = vrows[i]): dW_v = sum_t g_t (1[v=y_t] - exp(z_tv - lse_t)) h_t; 0 for v >= V_true.

    ``lse`` must hold the log-sum-exp of every token whose g is non-zero;
    tokens with g == 0 contribute nothing and their lse entry is not read.
    """
    kind, h, W = _pair(h, W)
    y = np.ascontiguousarray(y, dtype=np.int64)
    g = np.ascontiguousarray(g, dtype=np.float64)
    lse = np.ascontiguousarray(lse, dtype=np.float64)
    T, H = h.shape
    V = W.shape[0]
    if lse.shape != (T,):
        raise ValueError("lse must have one entry per token")
    r, n = _rows(vrows, V)
    dW = np.empty((n, H), np.float64)
    _check(_load().rlko_backward_dw(kind, _ptr(h), _ptr(W), _ptr(y), _ptr(g), _ptr(lse), T, H, V,
                                    int(V_true), _ptr(r), n, _ptr(dW), int(nthreads)),
           "rlko_backward_dw")
    return dW


def e4m3_to_double(code: int) -> float:
    """Value of one OCP E4M3 code (sign, 4 exponent bits with bias 7, 3 mantissa bits;
    no infinities, S.1111.111 = NaN)."""
    return float(_load().rlko_e4m3_to_double(int(code) & 0xFF))


def quantize_rows_e4m3(x, nthreads=0):
    """Per-row power-of-two scale and E4M3 codes of x (float64, or uint16 bf16 bits):
    e = the smallest integer with max|x_row| <= 448 * 2^e (0 for an all-zero row),
    code = the E4M3 value nearest to x / 2^e, ties to the even code.
    Returns (codes uint8 [rows, cols], scale float64 [rows] = 2^e)."""
    o = _Operand(x)
    if o.kind == E4M3:
        raise TypeError("quantize_rows_e4m3 takes float64 or bf16 bits")
    rows, cols = o.shape
    q = np.empty((rows, cols), np.uint8)
    scale = np.empty(rows, np.float64)
    _check(_load().rlko_quantize_rows_e4m3(o.kind, o.ptr, rows, cols, _ptr(q), _ptr(scale),
                                           int(nthreads)), "rlko_quantize_rows_e4m3")
    return q, scale


def backward_dh_ste(zh, zW, h, W, y, g, V_true, rows=None, nthreads=0):
    """Straight-through dH rows: p and dz from the logits of (zh, zW) (e.g. E4M3 operands),
    dH_t = sum_v dz_tv W_v with the unquantized W."""
    zk, zh, zW = _pair(zh, zW)
    kind, h, W = _pair(h, W)
    if zh.shape != h.shape or zW.shape != W.shape:
        raise ValueError("logit and gradient operands must have the same shapes")
    y = np.ascontiguousarray(y, dtype=np.int64)
    g = np.ascontiguousarray(g, dtype=np.float64)
    T, H = h.shape
    V = W.shape[0]
    r, n = _rows(rows, T)
    dH = np.empty((n, H), np.float64)
    _check(_load().rlko_backward_dh_ste(zk, _ptr(zh), _ptr(zW), kind, _ptr(h), _ptr(W), _ptr(y),
                                        _ptr(g), T, H, V, int(V_true), _ptr(r), n, _ptr(dH),
                                        int(nthreads)), "rlko_backward_dh_ste")
    return dH


def backward_dw_ste(zh, zW, h, y, g, lse, V_true, vrows=None, nthreads=0):
    """Straight-through dW rows: dz from the logits of (zh, zW) and the given lse,
    dW_v = sum_t dz_tv h_t with the unquantized h; 0 for v >= V_true."""
    zk, zh, zW = _pair(zh, zW)
    oh = _Operand(h)
    if zh.shape != oh.shape:
        raise ValueError("logit and gradient operands must have the same shapes")
    y = np.ascontiguousarray(y, dtype=np.int64)
    g = np.ascontiguousarray(g, dtype=np.float64)
    lse = np.ascontiguousarray(lse, dtype=np.float64)
    T, H = oh.shape
    V = zW.shape[0]
    if lse.shape != (T,):
        raise ValueError("lse must have one entry per token")
    r, n = _rows(vrows, V)
    dW = np.empty((n, H), np.float64)
    _check(_load().rlko_backward_dw_ste(zk, _ptr(zh), _ptr(zW), oh.kind, _ptr(oh), _ptr(y),
                                        _ptr(g), _ptr(lse), T, H, V, int(V_true), _ptr(r), n,
                                        _ptr(dW), int(nthreads)), "rlko_backward_dw_ste")
    return dW
