"""The debug-checks build of the library (device-side index and tensor-copy coordinate
checks, RLK_DEBUG_CHECKS=1; compute-sanitizer is not available here, so the kernels check
their own accesses and report a failed check through the error flag instead of trapping).

Every entry point runs through both builds on ragged shapes: the checked build raises no
flag and gives the plain build's results bit for bit. Then the bounds self-test makes one
check fail on purpose (the kernels are told the statistics workspace is one entry shorter
than it is; every access stays inside the real buffer) and the flag must report it, with
the context still usable afterwards.
"""
import numpy as np
import pytest
import torch

import workloads
from gpu_util import dev, dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rlk():
    from deterministic_token_logprob_gb300 import build
    build.build()
    build.build(debug_checks=True)
    import deterministic_token_logprob_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def _run_all(rlk, T, H, V, Vt, seed):
    """Every entry point once on one shape; returns (outputs, error flag)."""
    d = workloads.make_inputs(workloads.Workload("dbg", T=T, H=H, V=V, V_true=Vt, seed=seed))
    h, W, y, g = dev_bf16(d["h"]), dev_bf16(d["W"]), dev(d["y"]), dev(d["g"])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = {}
    out["logp"], out["lse"] = rlk.linear_logp_fwd(h, W, y, Vt, err_flag=err)
    out["dH"], out["dW"] = rlk.linear_logp_bwd(h, W, y, out["lse"], g, Vt, err_flag=err)
    (_, _), z = rlk.linear_logp_fwd_save(h, W, y, Vt, err_flag=err)
    out["dH_saved"], out["dW_saved"] = rlk.linear_logp_bwd_saved(h, W, y, out["lse"], g, z, Vt,
                                                                 err_flag=err)
    (_, _), p = rlk.linear_logp_fwd_save_probs(h, W, y, Vt, err_flag=err)
    out["dH_probs"], out["dW_probs"] = rlk.linear_logp_bwd_saved_probs(h, W, y, out["lse"], g, p, Vt,
                                                                       err_flag=err)
    parts, dHp = [], []
    bounds = rlk.shard_bounds(V, Vt, 2)
    if any(n == 0 for _, n in bounds):   # a small vocabulary leaves the second shard empty
        bounds = []
    for a, n in bounds:
        parts.append(rlk.linear_logp_fwd(h, W[a:a + n], y, Vt, vocab_start=a, partial=True,
                                         err_flag=err))
        ws = torch.empty(rlk.bwd_workspace_bytes(T, H, n), dtype=torch.uint8, device="cuda")
        dh = torch.empty((T, H), dtype=torch.float32, device="cuda")
        for st in (rlk.RLK_BWD_DZ, rlk.RLK_BWD_DH):
            rlk.linear_logp_bwd(h, W[a:a + n], y, out["lse"], g, Vt, vocab_start=a,
                                dH_fp32_partial=True, want_dW=False, out=(dh, None), workspace=ws,
                                stages=st, err_flag=err)
        dHp.append(dh)
    if bounds:
        out["merged_logp"], _ = rlk.lse_merge(torch.stack(parts))
        out["dH_sharded"] = rlk.shard_sum_bf16(torch.stack(dHp))
    if H % 16 == 0:
        hq, hs = rlk.quantize_rows_e4m3(h, err_flag=err)
        Wq, Ws = rlk.quantize_rows_e4m3(W, err_flag=err)
        out["logp8"], lse8 = rlk.linear_logp_fwd_fp8(hq, hs, Wq, Ws, y, Vt, err_flag=err)
        out["dH8"], out["dW8"] = rlk.linear_logp_bwd_fp8(h, W, hq, hs, Wq, Ws, y, lse8, g, Vt,
                                                         err_flag=err)
    torch.cuda.synchronize()
    return out, int(err.item())


@pytest.mark.parametrize("shape", [(7, 136, 1100, 1030), (129, 200, 2500, 2345),
                                   (300, 512, 70000, 69000)])
def test_checked_build_raises_no_flag_and_gives_the_same_bits(rlk, shape):
    from deterministic_token_logprob_gb300 import build
    T, H, V, Vt = shape
    with rlk.library(build.DEBUG_LIB):
        assert rlk.debug_checks()
        dbg, flag = _run_all(rlk, T, H, V, Vt, seed=T)
    assert not rlk.debug_checks()
    rel, rel_flag = _run_all(rlk, T, H, V, Vt, seed=T)
    assert flag == 0 and rel_flag == 0, (flag, rel_flag)
    assert dbg.keys() == rel.keys()
    for k in rel:
        assert torch.equal(dbg[k], rel[k]), k


def test_bounds_self_test_reports_a_failed_check(rlk):
    from deterministic_token_logprob_gb300 import build
    T, H, V, Vt = 300, 256, 5000, 4900
    d = workloads.make_inputs(workloads.Workload("dbgst", T=T, H=H, V=V, V_true=Vt, seed=3))
    h, W, y = dev_bf16(d["h"]), dev_bf16(d["W"]), dev(d["y"])
    with rlk.library(build.DEBUG_LIB):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        rlk.selftest_bounds_check(h, W, y, Vt, err)
        torch.cuda.synchronize()
        assert int(err.item()) & rlk.RLK_FLAG_BOUNDS
        # the context stays usable, and a normal call raises no flag
        err.zero_()
        logp, _ = rlk.linear_logp_fwd(h, W, y, Vt, err_flag=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0 and np.all(np.isfinite(logp.cpu().numpy()))
    # the plain build refuses the self-test
    with pytest.raises(rlk.RlkError):
        rlk.selftest_bounds_check(h, W, y, Vt, torch.zeros(1, dtype=torch.int32, device="cuda"))
