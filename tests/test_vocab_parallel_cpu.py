"""The cross-rank exchange of vocab-parallel linear_logp (deterministic_token_logprob_gb300.
vocab_parallel) on CPU: 2, 4 and 8 gloo ranks.

The exchange must hand the merge and the dH sum exactly the inputs the single-process
emulation gives them (the shards' statistics stacked in vocab order; the dH partials summed
in ascending shard order), bit for bit: then the merged logp / lse and the summed dH are the
emulation's bits, which the GPU tests compare with the unsharded call. The merge and the dH
sum themselves run on the GPU; here the statistics come from the oracle and the fixed-order
fp32 sum plus one bf16 rounding is done by torch on the host.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import workloads


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _host_sum_bf16(parts: torch.Tensor) -> torch.Tensor:
    """((p0 + p1) + p2) + ... in fp32 round-to-nearest, then one round-to-nearest-even to bf16."""
    acc = parts[0].clone()
    for i in range(1, parts.shape[0]):
        acc = acc + parts[i]
    return acc.to(torch.bfloat16)


def _stats_tensor(oracle, h, W, y, start, n, V_true):
    m, s, zt = oracle.shard_stats(h, W[start:start + n], y, start, V_true)
    return torch.from_numpy(np.stack([m, s, zt], axis=1).astype(np.float32))


def _partial(rank, T, H):
    return torch.from_numpy(np.random.default_rng(100 + rank).standard_normal((T, H)).astype(np.float32))


def _worker(rank, world, port, out):
    import torch.distributed as dist

    import oracle
    from deterministic_token_logprob_gb300 import _binding as rlk
    from deterministic_token_logprob_gb300 import vocab_parallel as vp
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        oracle.build()
        T, H, V, Vt = 37, 64, 6000, 5900
        w = workloads.Workload("vp", T=T, H=H, V=V, V_true=Vt, seed=5)
        d = workloads.make_inputs(w)
        bounds = rlk.shard_bounds(V, Vt, world)
        start, n = vp.shard_of_rank(V, Vt)
        assert (start, n) == bounds[rank]
        # forward: every rank's statistics, gathered in rank (= vocab) order
        mine = _stats_tensor(oracle, d["h"], d["W"], d["y"], start, n, Vt)
        got = vp.gather_stats(mine)
        emul = torch.stack([_stats_tensor(oracle, d["h"], d["W"], d["y"], a, k, Vt) for a, k in bounds])
        fwd_bitwise = torch.equal(got.view(torch.int32), emul.view(torch.int32))
        # the gathered statistics merge to the full forward (oracle merge, fp64)
        m, s, zt = (got[:, :, i].double().numpy() for i in range(3))
        logp, _ = oracle.lse_merge(m, s, zt)
        ref_logp, _ = oracle.forward(d["h"], d["W"], d["y"], Vt)
        fwd_err = float(np.max(np.abs(logp - ref_logp)))
        # backward: the fixed-order sum of the fp32 dH partials, ragged row counts included
        res = {}
        for Tb in (T, 1, 2, 8):
            dh = vp.sum_dH_partials(_partial(rank, Tb, 24), sum_fn=_host_sum_bf16)
            ref = _host_sum_bf16(torch.stack([_partial(r, Tb, 24) for r in range(world)]))
            res[Tb] = (tuple(dh.shape), dh.dtype == torch.bfloat16,
                       torch.equal(dh.view(torch.int16), ref.view(torch.int16)),
                       dh.view(torch.int16).numpy().tobytes())
        # an empty batch: no collective is entered, empty results of the right shapes
        empty = (tuple(vp.gather_stats(torch.empty((0, 3))).shape),
                 tuple(vp.sum_dH_partials(torch.empty((0, 24)), sum_fn=_host_sum_bf16).shape))
        out[rank] = (fwd_bitwise, fwd_err, res, empty)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4, 8])
def test_vocab_parallel_exchange_matches_single_process(world):
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert set(res) == set(range(world))
    for r in range(world):
        fwd_bitwise, fwd_err, sums, empty = res[r]
        assert empty == ((world, 0, 3), (0, 24))
        assert fwd_bitwise, f"rank {r}: gathered statistics differ from the vocab-order stack"
        assert fwd_err < 1e-5, fwd_err     # fp32-rounded statistics merged in fp64
        for Tb, (shape, is_bf16, same, _) in sums.items():
            assert shape == (Tb, 24) and is_bf16 and same, (r, Tb)
    for Tb in res[0][2]:       # every rank ends with the same dH
        assert len({res[r][2][Tb][3] for r in range(world)}) == 1


def test_shard_of_rank_requires_a_supported_group_size():
    from deterministic_token_logprob_gb300 import _binding as rlk
    with pytest.raises(ValueError):
        rlk.shard_bounds(151936, 151669, 3)
    # two ranks split at the super-shard boundary, as the emulated Qwen3-30B workload does
    assert rlk.shard_bounds(151936, 151669, 2) == list(workloads.QWEN3_30B_TP2.shards)


def _worker_small_vocab(rank, world, port, out):
    # linear_logp_fwd_tp / linear_logp_bwd_tp end to end on CPU ranks, with the library's calls
    # replaced by stand-ins (the oracle's shard statistics and merge, seeded fp32 dH partials),
    # for a vocabulary so small that some ranks hold no rows
    import torch.distributed as dist

    import oracle
    from deterministic_token_logprob_gb300 import _binding
    from deterministic_token_logprob_gb300 import vocab_parallel as vp
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        oracle.build()
        T, H, V, Vt = 9, 32, 3000, 2900
        d = workloads.make_inputs(workloads.Workload("vps", T=T, H=H, V=V, V_true=Vt, seed=8))
        calls = []

        def bits(t):
            return t.view(torch.int16).numpy().view(np.uint16)

        def fake_fwd(h, W, y, V_true, vocab_start=0, partial=False, **kw):
            calls.append("fwd")
            m, s, zt = oracle.shard_stats(bits(h), bits(W), y.numpy(), vocab_start, V_true)
            return torch.from_numpy(np.stack([m, s, zt], axis=1).astype(np.float32))

        def fake_merge(parts, **kw):
            p = parts.double().numpy()
            logp, lse = oracle.lse_merge(p[:, :, 0], p[:, :, 1], p[:, :, 2])
            return torch.from_numpy(logp.astype(np.float32)), torch.from_numpy(lse.astype(np.float32))

        def fake_bwd(h, W, y, lse, g, V_true, vocab_start=0, want_dW=True, **kw):
            calls.append("bwd")
            return _partial(rank, h.shape[0], h.shape[1]), torch.zeros((W.shape[0], h.shape[1]))

        _binding.linear_logp_fwd = fake_fwd
        _binding.lse_merge = fake_merge
        _binding.linear_logp_bwd = fake_bwd
        _binding.shard_sum_bf16 = _host_sum_bf16
        start, n = vp.shard_of_rank(V, Vt)
        h = torch.from_numpy(d["h"].view(np.int16)).view(torch.bfloat16)
        W = torch.from_numpy(d["W"][start:start + n].view(np.int16)).view(torch.bfloat16)
        y, g = torch.from_numpy(d["y"]), torch.from_numpy(d["g"])
        logp, lse = vp.linear_logp_fwd_tp(h, W, y, Vt, V)
        dH, dW = vp.linear_logp_bwd_tp(h, W, y, lse, g, Vt, V)
        ref_logp, _ = oracle.forward(d["h"], d["W"], d["y"], Vt)
        sizes = [k for _, k in _binding.shard_bounds(V, Vt, world)]
        parts = [(_partial(r, T, H) if sizes[r] else torch.zeros((T, H))) for r in range(world)]
        ref_dH = _host_sum_bf16(torch.stack(parts))
        out[rank] = (n, calls, float(np.max(np.abs(logp.double().numpy() - ref_logp))),
                     torch.equal(dH.view(torch.int16), ref_dH.view(torch.int16)), tuple(dW.shape))
    finally:
        dist.destroy_process_group()


def test_ranks_without_vocabulary_rows_take_part_in_the_exchange():
    world = 4
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker_small_vocab, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    sizes = [res[r][0] for r in range(world)]
    assert sizes[0] > 0 and 0 in sizes, sizes      # this vocabulary leaves some ranks empty
    for r in range(world):
        n, calls, err, dH_ok, dW_shape = res[r]
        assert calls == ([] if n == 0 else ["fwd", "bwd"]), (r, calls)   # empty: no library call
        assert err < 1e-5, (r, err)
        assert dH_ok, r
        assert dW_shape == (n, 32)
