"""Vocab-parallel linear_logp (deterministic_token_logprob_gb300.vocab_parallel) on the GPU
with a one-rank NCCL group: the collectives run on device buffers (all-gather of the
statistics, all-to-all and all-gather of the dH blocks), and the results equal the plain
unsharded calls bit for bit. Several ranks need several GPUs; their exchange is covered by
the gloo tests on CPU (tests/test_vocab_parallel_cpu.py) and the shard arithmetic by the
single-GPU sharded tests."""
import datetime
import socket

import pytest
import torch

import workloads
from gpu_util import dev, dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rlk():
    from deterministic_token_logprob_gb300 import build
    build.build()
    import deterministic_token_logprob_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_one_rank_group_equals_unsharded_calls(rlk):
    import torch.distributed as dist

    from deterministic_token_logprob_gb300 import vocab_parallel as vp
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{_free_port()}", rank=0,
                            world_size=1, timeout=datetime.timedelta(seconds=120))
    try:
        # V above 65536: dH reduces over two accumulation chunks
        for T, H, V, Vt in ((300, 256, 70000, 69000), (37, 128, 4096, 4000)):
            w = workloads.Workload("vp1", T=T, H=H, V=V, V_true=Vt, seed=9)
            d = workloads.make_inputs(w)
            h, W, y, g = dev_bf16(d["h"]), dev_bf16(d["W"]), dev(d["y"]), dev(d["g"])
            assert vp.shard_of_rank(V, Vt) == (0, V)
            logp, lse = vp.linear_logp_fwd_tp(h, W, y, Vt, V)
            dH, dW = vp.linear_logp_bwd_tp(h, W, y, lse, g, Vt, V)
            ref_logp, ref_lse = rlk.linear_logp_fwd(h, W, y, Vt)
            ref_dH, ref_dW = rlk.linear_logp_bwd(h, W, y, ref_lse, g, Vt)
            torch.cuda.synchronize()
            assert torch.equal(logp, ref_logp) and torch.equal(lse, ref_lse)
            assert dH.dtype == torch.bfloat16 and torch.equal(dH, ref_dH)
            assert torch.equal(dW, ref_dW)
    finally:
        dist.destroy_process_group()
