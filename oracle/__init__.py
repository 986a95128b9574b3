"""fp64 CPU oracle for `linear_logp` -- TEST INFRASTRUCTURE.

Only the test-suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. The product library never does, and this package
shares no code with it: the arithmetic lives in ``rlk_oracle.c`` (plain C99,
binary64), compiled by :func:`build` with gcc.

Inputs ``h`` and ``W`` are numpy arrays either of dtype float64 or of dtype
uint16 holding raw bf16 bit patterns (the exact values the GPU receives). Each
function states the definition it evaluates; the C file cites the passages.
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
            lib.rlko_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.rlko_bf16_to_double.restype = ctypes.c_double
            lib.rlko_default_threads.argtypes = []
            for name in ("rlko_forward", "rlko_shard_stats", "rlko_lse_merge",
                         "rlko_backward_dh", "rlko_backward_dw", "rlko_default_threads"):
                getattr(lib, name).restype = ctypes.c_int
            _lib = lib
    return _lib


def default_threads() -> int:
    """Number of host threads the oracle uses when nthreads=0 (all online cores)."""
    return int(_load().rlko_default_threads())


def bf16_to_double(bits: int) -> float:
    return float(_load().rlko_bf16_to_double(int(bits) & 0xFFFF))


def _mat(a: np.ndarray):
    if a.dtype == np.float64:
        return F64, np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return BF16, np.ascontiguousarray(a)
    raise TypeError(f"oracle inputs must be float64 or uint16 (bf16 bits), got {a.dtype}")


def _pair(h: np.ndarray, W: np.ndarray):
    dh, h = _mat(h)
    dw, W = _mat(W)
    if dh != dw:
        raise TypeError("h and W must have the same element kind")
    if h.ndim != 2 or W.ndim != 2 or h.shape[1] != W.shape[1]:
        raise ValueError(f"shape mismatch h{h.shape} W{W.shape}")
    return dh, h, W


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


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
