"""Vocab (tensor) parallelism across processes: the exchange between ranks of linear_logp.

Each rank of a process group holds the same tokens and one contiguous block of LM-head
rows: shard ``shard_bounds(V, V_true, S)[rank]`` of the fixed merge tree, S = the group's
size (1, 2, 4 or 8; the group rank is the shard index, so rank order is vocab order). Only
per-token statistics and gradient partials cross ranks. Each rank reduces its own vocabulary
shard and the ranks combine only the statistics the global selected log-probability needs
("Announcing RL-Kernel for vime", section "Why the Fused Path Wins", third reason), with a
local reduction per rank and a merge of the log-sum-exp statistics across ranks ("vLLM
RL-Kernel v0.1.0: Bitwise Train-Rollout Consistency on ROCm", table "Boundary Fixes in the
RL-Kernel Strict Path", row "Linear logprob").

forward   every rank: its shard's (m, s, zt) per token (rlk_linear_logp_fwd with a partial
          output); an all-gather of the [T, 3] triples into [S, T, 3] in rank order; every
          rank merges them with rlk_lse_merge (the top levels of the fixed tree), so all ranks
          hold the same logp and lse.
backward  every rank: its shard's fp32 dH partial and its own dW rows (rlk_linear_logp_bwd
          with the global lse; dW never leaves the rank). The dH partials are summed in
          ascending rank order and rounded once to bf16: an all-to-all hands rank r block r of
          the token rows of every rank's partial ([S, rows, H], rank order), rank r sums its
          block (rlk_shard_sum_bf16), and an all-gather of the bf16 blocks gives every rank dH.

No collective here adds numbers. An all-reduce sums in an order that belongs to the
communication library (and can change with the algorithm it picks for a message size), which
would break the bitwise contract; an all-gather and an all-to-all only move bytes, and every
sum runs in this library's fixed order. The results are therefore bit-identical to the
single-process emulation (the S shards one after another on one device, then rlk_lse_merge /
rlk_shard_sum_bf16), whose logp and lse are in turn bit-identical to the unsharded call.

Per rank and call, the bytes that cross the links: (S - 1) * 12 B per token in the forward;
(S - 1) / S * T * H * 4 B sent by the all-to-all and (S - 1) / S * T * H * 2 B received by the
all-gather in the backward (an all-gather of whole fp32 partials would move (S - 1) * T * H * 4 B).
"""
from __future__ import annotations

from typing import Callable, Optional, Tuple

import torch
import torch.distributed as dist

from . import _binding as rlk


def shard_of_rank(V: int, V_true: int, group=None) -> Tuple[int, int]:
    """(vocab_start, V_local) of the calling rank's shard of V LM-head rows."""
    S = dist.get_world_size(group)
    return rlk.shard_bounds(V, V_true, S)[dist.get_rank(group)]


def gather_stats(partial: torch.Tensor, group=None) -> torch.Tensor:
    """All-gather of every rank's [T, 3] shard statistics into [S, T, 3], slot i = rank i's."""
    S = dist.get_world_size(group)
    T = partial.shape[0]
    out = torch.empty((S * T,) + tuple(partial.shape[1:]), dtype=partial.dtype, device=partial.device)
    if T:   # every rank holds the same tokens, so all ranks skip an empty batch together
        dist.all_gather_into_tensor(out, partial.contiguous(), group=group)
    return out.view((S,) + tuple(partial.shape))


def sum_dH_partials(part: torch.Tensor, group=None,
                    sum_fn: Optional[Callable[[torch.Tensor], torch.Tensor]] = None) -> torch.Tensor:
    """bf16 dH = round(((p_0 + p_1) + p_2) + ...) of every rank's fp32 [T, H] partial p_r,
    the sum in ascending rank order. ``sum_fn`` maps fp32 [S, rows, H] to bf16 [rows, H] in
    that order (default: rlk_shard_sum_bf16 on the device)."""
    if sum_fn is None:
        sum_fn = lambda parts: rlk.shard_sum_bf16(parts)  # noqa: E731
    S = dist.get_world_size(group)
    T, H = part.shape
    if T == 0:  # the same on every rank: no rank enters the collectives
        return torch.empty((0, H), dtype=torch.bfloat16, device=part.device)
    rows = -(-T // S)
    if rows * S != T:   # pad to S equal row blocks; padding rows are summed and discarded
        padded = torch.zeros((rows * S, H), dtype=part.dtype, device=part.device)
        padded[:T] = part
        part = padded
    blocks = torch.empty((S * rows, H), dtype=part.dtype, device=part.device)
    # rank r receives block r of every rank, in rank order
    dist.all_to_all_single(blocks, part.contiguous(), group=group)
    mine = sum_fn(blocks.view(S, rows, H))
    full = torch.empty((S * rows, H), dtype=mine.dtype, device=part.device)
    dist.all_gather_into_tensor(full, mine.contiguous(), group=group)
    return full[:T]


def linear_logp_fwd_tp(h: torch.Tensor, W_local: torch.Tensor, y: torch.Tensor, V_true: int,
                       V: int, *, group=None, err_flag: Optional[torch.Tensor] = None,
                       workspace: Optional[torch.Tensor] = None):
    """Forward across the group: (logp, lse), fp32 [T] each, the same on every rank.
    W_local holds this rank's rows shard_of_rank(V, V_true, group) of the V-row LM head."""
    start, n = shard_of_rank(V, V_true, group)
    if W_local.shape[0] != n:
        raise ValueError(f"rank's W shard has {W_local.shape[0]} rows, its shard has {n}")
    if n == 0:
        # a small vocabulary can leave a rank no rows: its statistics are the merge's identity
        # (m = -inf, s = 0, zt = -inf), which the merge passes over bit for bit
        part = torch.tensor([float("-inf"), 0.0, float("-inf")], dtype=torch.float32,
                            device=h.device).repeat(h.shape[0], 1)
    else:
        part = rlk.linear_logp_fwd(h, W_local, y, V_true, vocab_start=start, partial=True,
                                   err_flag=err_flag, workspace=workspace)
    return rlk.lse_merge(gather_stats(part, group))


def linear_logp_bwd_tp(h: torch.Tensor, W_local: torch.Tensor, y: torch.Tensor, lse: torch.Tensor,
                       g: torch.Tensor, V_true: int, V: int, *, group=None, want_dW: bool = True,
                       err_flag: Optional[torch.Tensor] = None,
                       workspace: Optional[torch.Tensor] = None):
    """Backward across the group, with lse from linear_logp_fwd_tp: (dH, dW_local). dH is bf16
    [T, H], the same on every rank; dW_local is fp32, this rank's rows only (or None)."""
    start, n = shard_of_rank(V, V_true, group)
    if W_local.shape[0] != n:
        raise ValueError(f"rank's W shard has {W_local.shape[0]} rows, its shard has {n}")
    if n == 0:  # no rows on this rank: a zero dH partial, no dW rows
        T, H = h.shape
        dHp = torch.zeros((T, H), dtype=torch.float32, device=h.device)
        dW = torch.empty((0, H), dtype=torch.float32, device=h.device) if want_dW else None
    else:
        dHp, dW = rlk.linear_logp_bwd(h, W_local, y, lse, g, V_true, vocab_start=start,
                                      dH_fp32_partial=True, want_dW=want_dW, err_flag=err_flag,
                                      workspace=workspace)
    return sum_dH_partials(dHp, group), dW
