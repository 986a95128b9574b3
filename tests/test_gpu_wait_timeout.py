"""Failure detection without a GPU fault: a kernel wait made to run out.

rlk_selftest_wait_timeout leaves one pipeline stage unfilled on purpose, so the
tensor-core issuer's first wait cannot complete. The kernel must give up after
its wait limit, report RLK_FLAG_TIMEOUT through the caller's device flag, and
leave the CUDA context usable: a normal forward right after it is correct."""
import time

import numpy as np
import pytest
import torch

import workloads
from gpu_util import assert_logp_close, dev, dev_bf16

pytestmark = pytest.mark.gpu


def test_bounded_wait_expires_and_context_stays_usable(oracle_mod):
    from deterministic_token_logprob_gb300 import build
    build.build()
    import deterministic_token_logprob_gb300 as rlk
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    w = workloads.TINY
    d = workloads.make_inputs(w)
    h, W, y = dev_bf16(d["h"]), dev_bf16(d["W"]), dev(d["y"])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.time()
    rlk.selftest_wait_timeout(h, W, y, w.V_true, err)
    torch.cuda.synchronize()            # raises if the context were lost
    elapsed = time.time() - t0
    assert int(err.item()) & rlk.RLK_FLAG_TIMEOUT
    assert 1.5 < elapsed < 60.0, elapsed
    err.zero_()
    logp, lse = rlk.linear_logp_fwd(h, W, y, w.V_true, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref_logp, _ = oracle_mod.forward(d["h"], d["W"], d["y"], w.V_true)
    assert_logp_close(logp.cpu().numpy(), ref_logp)
