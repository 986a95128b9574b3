"""rlk_linear_logp_fwd_noalloc: the forward for callers that cannot allocate
device memory (a runtime whose memory is fully reserved up front, or a loop that
must not let cudaMalloc synchronise the device). Its scratch is a fixed static
device array inside the library instead of a caller-provided workspace.

The test calls it through the C ABI several times in a row and compares each result
with the workspace entry point's output on the same inputs, bit for bit: both run
the same kernels with the same arithmetic, so any difference would be a fault of
the static scratch (stale contents, aliasing, a counter not reset). Two of the
calls have the same shape and different data, so the second reuses exactly the
scratch offsets the first wrote. It runs on its own in a fresh process as well as
after the rest of the suite (this file is collected last).
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from gpu_util import dev, dev_bf16

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20


@pytest.fixture(scope="module")
def rlk():
    from deterministic_token_logprob_gb300 import build
    build.build()
    import deterministic_token_logprob_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    lib = m.lib()
    P, I64 = ctypes.c_void_p, ctypes.c_int64
    lib.rlk_linear_logp_fwd_noalloc.argtypes = [P, P, P, I64, I64, I64, I64, I64, P, P, P, P, P]
    lib.rlk_linear_logp_fwd_noalloc.restype = ctypes.c_int
    return m


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(rlk, h, W, y, V_true, vocab_start=0, partial=False, err=None):
    T, H = h.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if partial:
        p = torch.empty((T, 3), dtype=torch.float32, device="cuda")
        logp = lse = None
    else:
        p = None
        logp = torch.empty(T, dtype=torch.float32, device="cuda")
        lse = torch.empty(T, dtype=torch.float32, device="cuda")
    st = rlk.lib().rlk_linear_logp_fwd_noalloc(_ptr(h), _ptr(W), _ptr(y), T, H, W.shape[0],
                                               vocab_start, V_true, _ptr(logp), _ptr(lse), _ptr(p),
                                               _ptr(err), stream)
    assert st == rlk.RLK_OK, st
    return p if partial else (logp, lse)


def _case(T, H, V, Vt, seed):
    d = workloads.make_inputs(workloads.Workload("na", T=T, H=H, V=V, V_true=Vt, seed=seed))
    return dev_bf16(d["h"]), dev_bf16(d["W"]), dev(d["y"])


def _same_bits(a, b):
    assert torch.isfinite(a).all()
    assert torch.equal(a, b)


def test_noalloc_matches_workspace_entry_point_bitwise(rlk):
    # calls in a row: two shapes, then the first shape again on other data (same scratch
    # offsets as the first call, new values)
    cases = [(_case(300, 512, 20480, 20000, seed=41), 20000),
             (_case(1000, 256, 9000, 8999, seed=42), 8999),
             (_case(300, 512, 20480, 20000, seed=43), 20000)]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for (h, W, y), Vt in cases:
        ref_logp, ref_lse = rlk.linear_logp_fwd(h, W, y, Vt)
        logp, lse = _noalloc(rlk, h, W, y, Vt, err=err)
        torch.cuda.synchronize()
        _same_bits(logp, ref_logp)
        _same_bits(lse, ref_lse)
    assert int(err.item()) == 0
    # shard statistics through the same scratch, each against the workspace entry point's
    # statistics of the same shard, then the merge
    (h, W, y), Vt = cases[2]
    bounds = rlk.shard_bounds(20480, 20000, 2)
    parts = []
    for a, n in bounds:
        p = _noalloc(rlk, h, W[a:a + n], y, Vt, vocab_start=a, partial=True)
        ref = rlk.linear_logp_fwd(h, W[a:a + n], y, Vt, vocab_start=a, partial=True)
        torch.cuda.synchronize()
        assert torch.equal(p, ref)
        parts.append(p)
    logp, lse = rlk.lse_merge(torch.stack(parts))
    ref_logp, ref_lse = rlk.linear_logp_fwd(h, W, y, Vt)
    torch.cuda.synchronize()
    _same_bits(logp, ref_logp)
    _same_bits(lse, ref_lse)


def test_noalloc_rejects_shapes_beyond_its_scratch(rlk):
    lib = rlk.lib()
    V = 151936
    assert lib.rlk_linear_logp_fwd_workspace(9383, 4096, V) <= SCRATCH_BYTES
    assert lib.rlk_linear_logp_fwd_workspace(9384, 4096, V) > SCRATCH_BYTES
    fake = ctypes.c_void_p(0x100000)
    st = lib.rlk_linear_logp_fwd_noalloc(fake, fake, fake, 9384, 4096, V, 0, 151669, fake, fake,
                                         None, None, None)
    assert st == rlk.RLK_ERR_WORKSPACE
