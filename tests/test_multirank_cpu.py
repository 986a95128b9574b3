"""The multi-GPU (replica) path of bench.py on CPU: two gloo ranks.

Ranks run independent batches (token/data parallel: rows are independent and
batch-invariant, so there is no collective on the data path); the job's time
is the slowest rank's and its throughput counts every rank's tokens."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import workloads


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        elapsed = 100.0 + 25.0 * rank                  # rank 1 is the slow one
        mx = bench.max_over_ranks(elapsed, world)
        w = bench.rank_workload(workloads.TINY, rank)
        h = workloads.make_h(w.T, w.H, w.seed)
        digest = float(np.abs(workloads.bf16_to_f32(h)).sum())
        gathered = [None] * world
        dist.all_gather_object(gathered, digest)
        dist.barrier()
        out[rank] = (mx, w.seed, gathered,
                     bench.job_tokens_per_s(w.T, world, 10, mx))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_replicas():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 125.0                  # max over ranks
    assert res[0][1] == 0 and res[1][1] == 1                # each rank its own batch
    g0, g1 = res[0][2]
    assert g0 != g1                                         # ... so the batches differ
    assert res[0][2] == res[1][2]
    # whole-job throughput: both ranks' tokens over the slowest rank's time
    assert res[0][3] == pytest.approx(64 * 2 * 10 / 0.125)


def test_weight_is_shared_between_ranks():
    a = workloads.make_W(300, 64, seed=0)
    b = workloads.make_W(300, 64, seed=0)
    assert np.array_equal(a, b)
    w0 = bench_rank(0)
    w1 = bench_rank(1)
    assert not np.array_equal(workloads.make_h(w0.T, w0.H, w0.seed), workloads.make_h(w1.T, w1.H, w1.seed))


def bench_rank(rank):
    import bench
    return bench.rank_workload(workloads.TINY, rank)
