"""ctypes binding of librlk.so (include/rlk.h): argument marshalling only.

Every function here checks tensor placement, dtype and contiguity, allocates
the outputs and scratch the caller did not pass (through torch's allocator),
and calls the C entry point of the same name on the current torch stream. All
arithmetic runs in the library's CUDA kernels; there is no fallback path: if
librlk.so is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading
from typing import Optional, Sequence, Tuple

import torch

RLK_OK = 0
RLK_ERR_INVALID_ARG = 1
RLK_ERR_UNSUPPORTED = 2
RLK_ERR_WORKSPACE = 3
RLK_ERR_CUDA = 4

RLK_FLAG_BAD_TARGET = 1
RLK_FLAG_TIMEOUT = 2
RLK_FLAG_NONFINITE = 4
RLK_FLAG_BOUNDS = 8

RLK_BWD_DZ = 1
RLK_BWD_DH = 2
RLK_BWD_DW = 4

LEAF_WIDTH = 1024
MAX_SHARDS = 8

_PKG = os.path.dirname(os.path.abspath(__file__))
_lib = None
_lock = threading.Lock()


class RlkError(RuntimeError):
    def __init__(self, name: str, status: int):
        self.status = status
        msg = _load().rlk_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{name} returned {status} ({msg})")


def library_path() -> str:
    return os.path.join(_PKG, "_build", "librlk.so")


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"librlk.so is not built ({path}); run "
                               "`python -m deterministic_token_logprob_gb300.build`")
        _lib = _declare(ctypes.CDLL(path))
        return _lib


def _declare(lib):
    """Argument and result types of every entry point of include/rlk.h on a loaded library."""
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    lib.rlk_linear_logp_fwd_workspace.argtypes = [I64, I64, I64]
    lib.rlk_linear_logp_fwd_workspace.restype = SZ
    lib.rlk_linear_logp_bwd_workspace.argtypes = [I64, I64, I64]
    lib.rlk_linear_logp_bwd_workspace.restype = SZ
    lib.rlk_linear_logp_fwd.argtypes = [P, P, P, I64, I64, I64, I64, I64, P, P, P, P, P, SZ, P]
    lib.rlk_linear_logp_fwd.restype = ctypes.c_int
    lib.rlk_lse_merge.argtypes = [P, I32, I64, P, P, P]
    lib.rlk_lse_merge.restype = ctypes.c_int
    lib.rlk_linear_logp_bwd.argtypes = [P, P, P, P, P, I64, I64, I64, I64, I64, P, I32, P, P,
                                        P, SZ, P]
    lib.rlk_linear_logp_bwd.restype = ctypes.c_int
    lib.rlk_linear_logp_bwd_stages.argtypes = [P, P, P, P, P, I64, I64, I64, I64, I64, P, I32, P,
                                               I32, P, P, SZ, P]
    lib.rlk_linear_logp_bwd_stages.restype = ctypes.c_int
    lib.rlk_saved_logits_bytes.argtypes = [I64, I64]
    lib.rlk_saved_logits_bytes.restype = SZ
    lib.rlk_linear_logp_fwd_save.argtypes = [P, P, P, I64, I64, I64, I64, I64, P, P, P, P, SZ,
                                             P, P, SZ, P]
    lib.rlk_linear_logp_fwd_save.restype = ctypes.c_int
    lib.rlk_linear_logp_bwd_saved.argtypes = [P, P, P, P, P, P, SZ, I64, I64, I64, I64, I64, P,
                                              I32, P, P, P, SZ, P]
    lib.rlk_linear_logp_bwd_saved.restype = ctypes.c_int
    lib.rlk_saved_probs_bytes.argtypes = [I64, I64]
    lib.rlk_saved_probs_bytes.restype = SZ
    lib.rlk_linear_logp_fwd_save_probs.argtypes = [P, P, P, I64, I64, I64, I64, I64, P, P, P, P,
                                                   SZ, P, P, SZ, P]
    lib.rlk_linear_logp_fwd_save_probs.restype = ctypes.c_int
    lib.rlk_linear_logp_bwd_saved_probs.argtypes = [P, P, P, P, P, P, SZ, I64, I64, I64, I64,
                                                    I64, P, I32, P, P, P, SZ, P]
    lib.rlk_linear_logp_bwd_saved_probs.restype = ctypes.c_int
    lib.rlk_selftest_wait_timeout.argtypes = [P, P, P, I64, I64, I64, I64, P, P, P, P, SZ, P]
    lib.rlk_selftest_wait_timeout.restype = ctypes.c_int
    lib.rlk_shard_sum_bf16.argtypes = [P, I32, I64, P, P]
    lib.rlk_shard_sum_bf16.restype = ctypes.c_int
    lib.rlk_quantize_rows_e4m3.argtypes = [P, I64, I64, P, P, P, P]
    lib.rlk_quantize_rows_e4m3.restype = ctypes.c_int
    lib.rlk_linear_logp_fwd_fp8.argtypes = [P, P, P, P, P, I64, I64, I64, I64, I64, P, P, P, P,
                                            P, SZ, P]
    lib.rlk_linear_logp_fwd_fp8.restype = ctypes.c_int
    lib.rlk_linear_logp_bwd_fp8.argtypes = [P, P, P, P, P, P, P, P, P, I64, I64, I64, I64, I64,
                                            P, I32, P, P, P, SZ, P]
    lib.rlk_linear_logp_bwd_fp8.restype = ctypes.c_int
    lib.rlk_status_string.argtypes = [ctypes.c_int]
    lib.rlk_status_string.restype = ctypes.c_char_p
    lib.rlk_version.argtypes = []
    lib.rlk_version.restype = ctypes.c_char_p
    lib.rlk_debug_checks.argtypes = []
    lib.rlk_debug_checks.restype = ctypes.c_int32
    lib.rlk_selftest_bounds_check.argtypes = [P, P, P, I64, I64, I64, I64, P, P, P, P, SZ, P]
    lib.rlk_selftest_bounds_check.restype = ctypes.c_int
    return lib


@contextlib.contextmanager
def library(path: str):
    """Route every call of this module to the librlk.so at `path` (e.g. the debug-checks
    build) inside the `with` block; the library loaded before is restored afterwards."""
    global _lib
    other = _declare(ctypes.CDLL(path))
    with _lock:
        prev = _lib
        _lib = other
    try:
        yield other
    finally:
        with _lock:
            _lib = prev


def lib():
    """The loaded ctypes library (raises if it is not built)."""
    return _load()


def version() -> str:
    return _load().rlk_version().decode()


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, ndim: int):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _check(name: str, status: int):
    if status != RLK_OK:
        raise RlkError(name, status)


def fwd_workspace_bytes(T: int, H: int, V_local: int) -> int:
    return int(_load().rlk_linear_logp_fwd_workspace(T, H, V_local))


def bwd_workspace_bytes(T: int, H: int, V_local: int) -> int:
    return int(_load().rlk_linear_logp_bwd_workspace(T, H, V_local))


def _workspace(nbytes: int, device, workspace: Optional[torch.Tensor]) -> Optional[torch.Tensor]:
    if nbytes == 0:
        return workspace
    if workspace is None:
        return torch.empty(nbytes, dtype=torch.uint8, device=device)
    if workspace.numel() * workspace.element_size() < nbytes:
        raise ValueError(f"workspace too small: need {nbytes} bytes")
    return workspace


def linear_logp_fwd(h: torch.Tensor, W: torch.Tensor, y: torch.Tensor, V_true: int, *,
                    vocab_start: int = 0, partial: bool = False,
                    out: Optional[Sequence[torch.Tensor]] = None,
                    err_flag: Optional[torch.Tensor] = None,
                    workspace: Optional[torch.Tensor] = None, stream=None):
    """rlk_linear_logp_fwd.

    partial=False: returns (logp, lse), fp32 [T] each (the shard must cover
    [0, V_true)). partial=True: returns this shard's statistics as fp32 [T, 3]
    (m, s, zt per token), to be combined with :func:`lse_merge`.
    `out` optionally supplies the output tensors ((logp, lse) or (partial,)).
    """
    _need(h, "h", torch.bfloat16, 2)
    _need(W, "W", torch.bfloat16, 2)
    _need(y, "y", torch.int64, 1)
    T, H = h.shape
    V_local = W.shape[0]
    if W.shape[1] != H or y.shape[0] != T:
        raise ValueError("shape mismatch")
    dev = h.device
    ws = _workspace(fwd_workspace_bytes(T, H, V_local), dev, workspace)
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    if partial:
        p = out[0] if out is not None else torch.empty((T, 3), dtype=torch.float32, device=dev)
        _need(p, "partial", torch.float32, 2)
        logp = lse = None
    else:
        p = None
        if out is not None:
            logp, lse = out
        else:
            logp = torch.empty(T, dtype=torch.float32, device=dev)
            lse = torch.empty(T, dtype=torch.float32, device=dev)
        _need(logp, "logp", torch.float32, 1)
        _need(lse, "lse", torch.float32, 1)
    if err_flag is not None:
        _need(err_flag, "err_flag", torch.int32, 1)
    st = _load().rlk_linear_logp_fwd(_ptr(h), _ptr(W), _ptr(y), T, H, V_local, int(vocab_start),
                                     int(V_true), _ptr(logp), _ptr(lse), _ptr(p), _ptr(err_flag),
                                     _ptr(ws), nbytes, _stream_handle(stream))
    _check("rlk_linear_logp_fwd", st)
    return p if partial else (logp, lse)


def lse_merge(partials: torch.Tensor, *, out: Optional[Tuple[torch.Tensor, torch.Tensor]] = None,
              stream=None):
    """rlk_lse_merge over fp32 [S, T, 3] shard statistics -> (logp, lse)."""
    _need(partials, "partials", torch.float32, 3)
    S, T, three = partials.shape
    if three != 3:
        raise ValueError("partials must be [S, T, 3]")
    if out is not None:
        logp, lse = out
    else:
        logp = torch.empty(T, dtype=torch.float32, device=partials.device)
        lse = torch.empty(T, dtype=torch.float32, device=partials.device)
    st = _load().rlk_lse_merge(_ptr(partials), S, T, _ptr(logp), _ptr(lse), _stream_handle(stream))
    _check("rlk_lse_merge", st)
    return logp, lse


def linear_logp_bwd(h: torch.Tensor, W: torch.Tensor, y: torch.Tensor, lse: torch.Tensor,
                    g: torch.Tensor, V_true: int, *, vocab_start: int = 0,
                    dH_fp32_partial: bool = False, want_dH: bool = True, want_dW: bool = True,
                    out: Optional[Tuple[Optional[torch.Tensor], Optional[torch.Tensor]]] = None,
                    err_flag: Optional[torch.Tensor] = None,
                    workspace: Optional[torch.Tensor] = None, stages: Optional[int] = None,
                    stream=None):
    """rlk_linear_logp_bwd -> (dH, dW); dH bf16 [T, H] (fp32 if dH_fp32_partial), dW fp32 [V_local, H].

    stages (an OR of RLK_BWD_DZ / RLK_BWD_DH / RLK_BWD_DW) calls rlk_linear_logp_bwd_stages
    instead: only those stages run, and the dz they share lives in `workspace`, which the
    caller then passes, unchanged, to the calls of the later stages."""
    _need(h, "h", torch.bfloat16, 2)
    _need(W, "W", torch.bfloat16, 2)
    _need(y, "y", torch.int64, 1)
    _need(lse, "lse", torch.float32, 1)
    _need(g, "g", torch.float32, 1)
    T, H = h.shape
    V_local = W.shape[0]
    if W.shape[1] != H or y.shape[0] != T or lse.shape[0] != T or g.shape[0] != T:
        raise ValueError("shape mismatch")
    dev = h.device
    if out is not None:
        dH, dW = out
    else:
        dH = (torch.empty((T, H), dtype=torch.float32 if dH_fp32_partial else torch.bfloat16,
                          device=dev) if want_dH else None)
        dW = torch.empty((V_local, H), dtype=torch.float32, device=dev) if want_dW else None
    if dH is not None:
        _need(dH, "dH", torch.float32 if dH_fp32_partial else torch.bfloat16, 2)
    if dW is not None:
        _need(dW, "dW", torch.float32, 2)
    if err_flag is not None:
        _need(err_flag, "err_flag", torch.int32, 1)
    if stages is not None and workspace is None:
        raise ValueError("stages need a caller-owned workspace (it carries dz between the calls)")
    ws = _workspace(bwd_workspace_bytes(T, H, V_local), dev, workspace)
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    if stages is None:
        st = _load().rlk_linear_logp_bwd(_ptr(h), _ptr(W), _ptr(y), _ptr(lse), _ptr(g), T, H,
                                         V_local, int(vocab_start), int(V_true), _ptr(dH),
                                         1 if dH_fp32_partial else 0, _ptr(dW), _ptr(err_flag),
                                         _ptr(ws), nbytes, _stream_handle(stream))
        _check("rlk_linear_logp_bwd", st)
    else:
        st = _load().rlk_linear_logp_bwd_stages(_ptr(h), _ptr(W), _ptr(y), _ptr(lse), _ptr(g), T, H,
                                                V_local, int(vocab_start), int(V_true), _ptr(dH),
                                                1 if dH_fp32_partial else 0, _ptr(dW), int(stages),
                                                _ptr(err_flag), _ptr(ws), nbytes,
                                                _stream_handle(stream))
        _check("rlk_linear_logp_bwd_stages", st)
    return dH, dW


def saved_logits_bytes(T: int, V_local: int) -> int:
    return int(_load().rlk_saved_logits_bytes(T, V_local))


def saved_logits_buffer(T: int, V_local: int, device="cuda") -> torch.Tensor:
    """An fp32 [T, round_up(V_local, 256)] buffer for the saved-logits pair."""
    return torch.empty((T, -(-V_local // 256) * 256), dtype=torch.float32, device=device)


def linear_logp_fwd_save(h: torch.Tensor, W: torch.Tensor, y: torch.Tensor, V_true: int, *,
                         vocab_start: int = 0, partial: bool = False,
                         z_saved: Optional[torch.Tensor] = None,
                         out: Optional[Sequence[torch.Tensor]] = None,
                         err_flag: Optional[torch.Tensor] = None,
                         workspace: Optional[torch.Tensor] = None, stream=None):
    """rlk_linear_logp_fwd_save: the forward that also stores its fp32 logits.

    Returns ((logp, lse) or partial, z_saved).
    """
    _need(h, "h", torch.bfloat16, 2)
    _need(W, "W", torch.bfloat16, 2)
    _need(y, "y", torch.int64, 1)
    T, H = h.shape
    V_local = W.shape[0]
    if W.shape[1] != H or y.shape[0] != T:
        raise ValueError("shape mismatch")
    dev = h.device
    if z_saved is None:
        z_saved = saved_logits_buffer(T, V_local, dev)
    _need(z_saved, "z_saved", torch.float32, 2)
    ws = _workspace(fwd_workspace_bytes(T, H, V_local), dev, workspace)
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    if partial:
        p = out[0] if out is not None else torch.empty((T, 3), dtype=torch.float32, device=dev)
        _need(p, "partial", torch.float32, 2)
        logp = lse = None
    else:
        p = None
        if out is not None:
            logp, lse = out
        else:
            logp = torch.empty(T, dtype=torch.float32, device=dev)
            lse = torch.empty(T, dtype=torch.float32, device=dev)
    if err_flag is not None:
        _need(err_flag, "err_flag", torch.int32, 1)
    st = _load().rlk_linear_logp_fwd_save(
        _ptr(h), _ptr(W), _ptr(y), T, H, V_local, int(vocab_start), int(V_true), _ptr(logp),
        _ptr(lse), _ptr(p), _ptr(z_saved), z_saved.numel() * 4, _ptr(err_flag), _ptr(ws), nbytes,
        _stream_handle(stream))
    _check("rlk_linear_logp_fwd_save", st)
    return (p if partial else (logp, lse)), z_saved


def linear_logp_bwd_saved(h: torch.Tensor, W: torch.Tensor, y: torch.Tensor, lse: torch.Tensor,
                          g: torch.Tensor, z_saved: torch.Tensor, V_true: int, *,
                          vocab_start: int = 0, dH_fp32_partial: bool = False,
                          want_dH: bool = True, want_dW: bool = True,
                          out: Optional[Tuple[Optional[torch.Tensor], Optional[torch.Tensor]]] = None,
                          err_flag: Optional[torch.Tensor] = None,
                          workspace: Optional[torch.Tensor] = None, stream=None):
    """rlk_linear_logp_bwd_saved: the backward from the forward's saved logits -> (dH, dW)."""
    _need(h, "h", torch.bfloat16, 2)
    _need(W, "W", torch.bfloat16, 2)
    _need(y, "y", torch.int64, 1)
    _need(lse, "lse", torch.float32, 1)
    _need(g, "g", torch.float32, 1)
    _need(z_saved, "z_saved", torch.float32, 2)
    T, H = h.shape
    V_local = W.shape[0]
    dev = h.device
    if out is not None:
        dH, dW = out
    else:
        dH = (torch.empty((T, H), dtype=torch.float32 if dH_fp32_partial else torch.bfloat16,
                          device=dev) if want_dH else None)
        dW = torch.empty((V_local, H), dtype=torch.float32, device=dev) if want_dW else None
    if err_flag is not None:
        _need(err_flag, "err_flag", torch.int32, 1)
    ws = _workspace(bwd_workspace_bytes(T, H, V_local), dev, workspace)
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    st = _load().rlk_linear_logp_bwd_saved(
        _ptr(h), _ptr(W), _ptr(y), _ptr(lse), _ptr(g), _ptr(z_saved), z_saved.numel() * 4, T, H,
        V_local, int(vocab_start), int(V_true), _ptr(dH), 1 if dH_fp32_partial else 0, _ptr(dW),
        _ptr(err_flag), _ptr(ws), nbytes, _stream_handle(stream))
    _check("rlk_linear_logp_bwd_saved", st)
    return dH, dW


def saved_probs_bytes(T: int, V_local: int) -> int:
    return int(_load().rlk_saved_probs_bytes(T, V_local))


def linear_logp_fwd_save_probs(h: torch.Tensor, W: torch.Tensor, y: torch.Tensor, V_true: int, *,
                               vocab_start: int = 0, partial: bool = False,
                               p_saved: Optional[torch.Tensor] = None,
                               out: Optional[Sequence[torch.Tensor]] = None,
                               err_flag: Optional[torch.Tensor] = None,
                               workspace: Optional[torch.Tensor] = None, stream=None):
    """rlk_linear_logp_fwd_save_probs: the forward that also stores bf16 probabilities
    (and their fp32 chunk maxima) in one byte buffer. Returns ((logp, lse) or partial, p_saved)."""
    _need(h, "h", torch.bfloat16, 2)
    _need(W, "W", torch.bfloat16, 2)
    _need(y, "y", torch.int64, 1)
    T, H = h.shape
    V_local = W.shape[0]
    dev = h.device
    if p_saved is None:
        p_saved = torch.empty(max(1, saved_probs_bytes(T, V_local)), dtype=torch.uint8, device=dev)
    _need(p_saved, "p_saved", torch.uint8, 1)
    ws = _workspace(fwd_workspace_bytes(T, H, V_local), dev, workspace)
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    if partial:
        p = out[0] if out is not None else torch.empty((T, 3), dtype=torch.float32, device=dev)
        logp = lse = None
    else:
        p = None
        if out is not None:
            logp, lse = out
        else:
            logp = torch.empty(T, dtype=torch.float32, device=dev)
            lse = torch.empty(T, dtype=torch.float32, device=dev)
    st = _load().rlk_linear_logp_fwd_save_probs(
        _ptr(h), _ptr(W), _ptr(y), T, H, V_local, int(vocab_start), int(V_true), _ptr(logp),
        _ptr(lse), _ptr(p), _ptr(p_saved), p_saved.numel(), _ptr(err_flag), _ptr(ws), nbytes,
        _stream_handle(stream))
    _check("rlk_linear_logp_fwd_save_probs", st)
    return (p if partial else (logp, lse)), p_saved


def linear_logp_bwd_saved_probs(h: torch.Tensor, W: torch.Tensor, y: torch.Tensor,
                                lse: torch.Tensor, g: torch.Tensor, p_saved: torch.Tensor,
                                V_true: int, *, vocab_start: int = 0,
                                dH_fp32_partial: bool = False, want_dH: bool = True,
                                want_dW: bool = True,
                                out: Optional[Tuple[Optional[torch.Tensor], Optional[torch.Tensor]]] = None,
                                err_flag: Optional[torch.Tensor] = None,
                                workspace: Optional[torch.Tensor] = None, stream=None):
    """rlk_linear_logp_bwd_saved_probs: the backward from saved bf16 probabilities -> (dH, dW)."""
    _need(h, "h", torch.bfloat16, 2)
    _need(W, "W", torch.bfloat16, 2)
    _need(y, "y", torch.int64, 1)
    _need(lse, "lse", torch.float32, 1)
    _need(g, "g", torch.float32, 1)
    _need(p_saved, "p_saved", torch.uint8, 1)
    T, H = h.shape
    V_local = W.shape[0]
    dev = h.device
    if out is not None:
        dH, dW = out
    else:
        dH = (torch.empty((T, H), dtype=torch.float32 if dH_fp32_partial else torch.bfloat16,
                          device=dev) if want_dH else None)
        dW = torch.empty((V_local, H), dtype=torch.float32, device=dev) if want_dW else None
    ws = _workspace(bwd_workspace_bytes(T, H, V_local), dev, workspace)
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    st = _load().rlk_linear_logp_bwd_saved_probs(
        _ptr(h), _ptr(W), _ptr(y), _ptr(lse), _ptr(g), _ptr(p_saved), p_saved.numel(), T, H,
        V_local, int(vocab_start), int(V_true), _ptr(dH), 1 if dH_fp32_partial else 0, _ptr(dW),
        _ptr(err_flag), _ptr(ws), nbytes, _stream_handle(stream))
    _check("rlk_linear_logp_bwd_saved_probs", st)
    return dH, dW


def debug_checks() -> bool:
    """True when the loaded library was built with device-side index checks."""
    return bool(_load().rlk_debug_checks())


def selftest_bounds_check(h: torch.Tensor, W: torch.Tensor, y: torch.Tensor, V_true: int,
                          err_flag: torch.Tensor, stream=None) -> None:
    """rlk_selftest_bounds_check (debug-checks builds): a forward told that its statistics
    workspace is one entry short; afterwards err_flag holds RLK_FLAG_BOUNDS."""
    _need(h, "h", torch.bfloat16, 2)
    _need(W, "W", torch.bfloat16, 2)
    _need(y, "y", torch.int64, 1)
    _need(err_flag, "err_flag", torch.int32, 1)
    T, H = h.shape
    V = W.shape[0]
    ws = _workspace(fwd_workspace_bytes(T, H, V), h.device, None)
    logp = torch.empty(T, dtype=torch.float32, device=h.device)
    lse = torch.empty(T, dtype=torch.float32, device=h.device)
    st = _load().rlk_selftest_bounds_check(_ptr(h), _ptr(W), _ptr(y), T, H, V, int(V_true),
                                           _ptr(logp), _ptr(lse), _ptr(err_flag), _ptr(ws),
                                           ws.numel(), _stream_handle(stream))
    _check("rlk_selftest_bounds_check", st)


def selftest_wait_timeout(h: torch.Tensor, W: torch.Tensor, y: torch.Tensor, V_true: int,
                          err_flag: torch.Tensor, stream=None) -> None:
    """rlk_selftest_wait_timeout: a forward whose first pipeline wait is made to run
    out; afterwards (once the stream is synchronised) err_flag holds RLK_FLAG_TIMEOUT."""
    _need(h, "h", torch.bfloat16, 2)
    _need(W, "W", torch.bfloat16, 2)
    _need(y, "y", torch.int64, 1)
    _need(err_flag, "err_flag", torch.int32, 1)
    T, H = h.shape
    V = W.shape[0]
    ws = _workspace(fwd_workspace_bytes(T, H, V), h.device, None)
    logp = torch.empty(T, dtype=torch.float32, device=h.device)
    lse = torch.empty(T, dtype=torch.float32, device=h.device)
    st = _load().rlk_selftest_wait_timeout(_ptr(h), _ptr(W), _ptr(y), T, H, V, int(V_true),
                                           _ptr(logp), _ptr(lse), _ptr(err_flag), _ptr(ws),
                                           ws.numel(), _stream_handle(stream))
    _check("rlk_selftest_wait_timeout", st)


def shard_sum_bf16(partials: torch.Tensor, *, out: Optional[torch.Tensor] = None, stream=None):
    """rlk_shard_sum_bf16: fp32 [S, ...] -> bf16 [...], ascending-order sum, one rounding."""
    if not partials.is_cuda or partials.dtype != torch.float32 or not partials.is_contiguous():
        raise ValueError("partials must be a contiguous fp32 CUDA tensor [S, ...]")
    S = partials.shape[0]
    n = partials[0].numel()
    if out is None:
        out = torch.empty(partials.shape[1:], dtype=torch.bfloat16, device=partials.device)
    if out.dtype != torch.bfloat16 or not out.is_contiguous() or out.numel() != n:
        raise ValueError("out must be a contiguous bf16 tensor of one shard's shape")
    st = _load().rlk_shard_sum_bf16(_ptr(partials), S, n, _ptr(out), _stream_handle(stream))
    _check("rlk_shard_sum_bf16", st)
    return out


def shard_bounds(V: int, V_true: int, S: int):
    """(vocab_start, V_local) of S contiguous shards that the fixed merge tree can express.

    The tree groups ceil(V_true/1024) leaves into 8 super-shards of
    L = ceil(nLeaves/8) leaves; shard i of S covers super-shards
    [8i/S, 8(i+1)/S) and the last shard runs to V.
    """
    if S not in (1, 2, 4, 8):
        raise ValueError("S must be 1, 2, 4 or 8")
    n_leaves = -(-V_true // LEAF_WIDTH)
    width = -(-n_leaves // MAX_SHARDS) * LEAF_WIDTH
    per = MAX_SHARDS // S
    out = []
    for i in range(S):
        a = min(i * per * width, V)
        b = V if i == S - 1 else min((i + 1) * per * width, V)
        out.append((a, b - a))
    return out


# --------------------------------------------------------------------------- FP8 LM head


def quantize_rows_e4m3(x: torch.Tensor, *, out: Optional[Tuple[torch.Tensor, torch.Tensor]] = None,
                       err_flag: Optional[torch.Tensor] = None, stream=None):
    """rlk_quantize_rows_e4m3 -> (codes uint8 [rows, cols], scale fp32 [rows]).

    scale[r] = 2^e with e the smallest integer such that max|x[r]| <= 448 * 2^e;
    codes = E4M3(x / scale) rounded to nearest even.
    """
    _need(x, "x", torch.bfloat16, 2)
    rows, cols = x.shape
    if out is not None:
        q, scale = out
    else:
        q = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
        scale = torch.empty(rows, dtype=torch.float32, device=x.device)
    _need(q, "q", torch.uint8, 2)
    _need(scale, "scale", torch.float32, 1)
    if tuple(q.shape) != (rows, cols) or scale.shape[0] != rows:
        raise ValueError("shape mismatch")
    if err_flag is not None:
        _need(err_flag, "err_flag", torch.int32, 1)
    st = _load().rlk_quantize_rows_e4m3(_ptr(x), rows, cols, _ptr(q), _ptr(scale), _ptr(err_flag),
                                        _stream_handle(stream))
    _check("rlk_quantize_rows_e4m3", st)
    return q, scale


def linear_logp_fwd_fp8(hq: torch.Tensor, h_scale: torch.Tensor, Wq: torch.Tensor,
                        W_scale: torch.Tensor, y: torch.Tensor, V_true: int, *,
                        vocab_start: int = 0, partial: bool = False,
                        out: Optional[Sequence[torch.Tensor]] = None,
                        err_flag: Optional[torch.Tensor] = None,
                        workspace: Optional[torch.Tensor] = None, stream=None):
    """rlk_linear_logp_fwd_fp8 on E4M3 codes + per-row scales (from :func:`quantize_rows_e4m3`);
    returns as :func:`linear_logp_fwd`."""
    _need(hq, "hq", torch.uint8, 2)
    _need(Wq, "Wq", torch.uint8, 2)
    _need(h_scale, "h_scale", torch.float32, 1)
    _need(W_scale, "W_scale", torch.float32, 1)
    _need(y, "y", torch.int64, 1)
    T, H = hq.shape
    V_local = Wq.shape[0]
    if Wq.shape[1] != H or y.shape[0] != T or h_scale.shape[0] != T or W_scale.shape[0] != V_local:
        raise ValueError("shape mismatch")
    dev = hq.device
    ws = _workspace(fwd_workspace_bytes(T, H, V_local), dev, workspace)
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    if partial:
        p = out[0] if out is not None else torch.empty((T, 3), dtype=torch.float32, device=dev)
        _need(p, "partial", torch.float32, 2)
        logp = lse = None
    else:
        p = None
        if out is not None:
            logp, lse = out
        else:
            logp = torch.empty(T, dtype=torch.float32, device=dev)
            lse = torch.empty(T, dtype=torch.float32, device=dev)
        _need(logp, "logp", torch.float32, 1)
        _need(lse, "lse", torch.float32, 1)
    if err_flag is not None:
        _need(err_flag, "err_flag", torch.int32, 1)
    st = _load().rlk_linear_logp_fwd_fp8(_ptr(hq), _ptr(h_scale), _ptr(Wq), _ptr(W_scale), _ptr(y),
                                         T, H, V_local, int(vocab_start), int(V_true), _ptr(logp),
                                         _ptr(lse), _ptr(p), _ptr(err_flag), _ptr(ws), nbytes,
                                         _stream_handle(stream))
    _check("rlk_linear_logp_fwd_fp8", st)
    return p if partial else (logp, lse)


def linear_logp_bwd_fp8(h: torch.Tensor, W: torch.Tensor, hq: torch.Tensor, h_scale: torch.Tensor,
                        Wq: torch.Tensor, W_scale: torch.Tensor, y: torch.Tensor, lse: torch.Tensor,
                        g: torch.Tensor, V_true: int, *, vocab_start: int = 0,
                        dH_fp32_partial: bool = False, want_dH: bool = True, want_dW: bool = True,
                        out: Optional[Tuple[Optional[torch.Tensor], Optional[torch.Tensor]]] = None,
                        err_flag: Optional[torch.Tensor] = None,
                        workspace: Optional[torch.Tensor] = None, stream=None):
    """rlk_linear_logp_bwd_fp8 (straight-through): dz from the E4M3 logits, dH = dz W and
    dW = dz^T h with the bf16 operands; returns (dH, dW) as :func:`linear_logp_bwd`."""
    _need(h, "h", torch.bfloat16, 2)
    _need(W, "W", torch.bfloat16, 2)
    _need(hq, "hq", torch.uint8, 2)
    _need(Wq, "Wq", torch.uint8, 2)
    _need(h_scale, "h_scale", torch.float32, 1)
    _need(W_scale, "W_scale", torch.float32, 1)
    _need(y, "y", torch.int64, 1)
    _need(lse, "lse", torch.float32, 1)
    _need(g, "g", torch.float32, 1)
    T, H = h.shape
    V_local = W.shape[0]
    if (W.shape[1] != H or tuple(hq.shape) != (T, H) or tuple(Wq.shape) != (V_local, H)
            or y.shape[0] != T or lse.shape[0] != T or g.shape[0] != T
            or h_scale.shape[0] != T or W_scale.shape[0] != V_local):
        raise ValueError("shape mismatch")
    dev = h.device
    if out is not None:
        dH, dW = out
    else:
        dH = (torch.empty((T, H), dtype=torch.float32 if dH_fp32_partial else torch.bfloat16,
                          device=dev) if want_dH else None)
        dW = torch.empty((V_local, H), dtype=torch.float32, device=dev) if want_dW else None
    if dH is not None:
        _need(dH, "dH", torch.float32 if dH_fp32_partial else torch.bfloat16, 2)
    if dW is not None:
        _need(dW, "dW", torch.float32, 2)
    if err_flag is not None:
        _need(err_flag, "err_flag", torch.int32, 1)
    ws = _workspace(bwd_workspace_bytes(T, H, V_local), dev, workspace)
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    st = _load().rlk_linear_logp_bwd_fp8(_ptr(h), _ptr(W), _ptr(hq), _ptr(h_scale), _ptr(Wq),
                                         _ptr(W_scale), _ptr(y), _ptr(lse), _ptr(g), T, H, V_local,
                                         int(vocab_start), int(V_true), _ptr(dH),
                                         1 if dH_fp32_partial else 0, _ptr(dW), _ptr(err_flag),
                                         _ptr(ws), nbytes, _stream_handle(stream))
    _check("rlk_linear_logp_bwd_fp8", st)
    return dH, dW
