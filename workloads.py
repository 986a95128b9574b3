"""Seeded synthetic inputs for `linear_logp` -- shapes, distributions, seeds.

This module holds no arithmetic of the method: it only draws inputs (numpy
PCG64, seeded) and rounds them to bf16 bit patterns. Both the oracle (tests,
CPU baseline) and the GPU path (tests, bench, smoke) take their inputs from
here, so both sides see identical bits.

Workloads (shapes follow the Qwen3 output layers the pages benchmark on: the
"Announcing RL-Kernel for vime" validation section uses Qwen3-30B-A3B, the
RL-Kernel README's end-to-end path uses Qwen3-8B Dense):

* ``tiny``          T=64, H=256, V=V_true=4096; g ~ N(0,1).
* ``qwen3_8b_fwd``  T=4096, H=4096, V=151936, V_true=151669 (forward only).
* ``qwen3_8b``      T=8192 = 16 sequences x 512 tokens, same H/V; g is a
                    per-sequence GRPO-style advantage A_s ~ N(0,1) divided by
                    the sequence's token count (512).
* ``qwen3_30b_tp2`` T=16384 = 32 x 512, H=2048, same V; two contiguous vocab
                    shards [0, 77824) and [77824, 151936); g as above.
* ``invariance``    128 seeded (hidden, target) pairs at H=4096, V_true=151669,
                    embedded in ragged batches of T in {1, 7, 128, 1000, 4097}
                    among filler rows ~ N(0,1).

h ~ N(0,1) and W ~ N(0, 0.02) are drawn in float32 and rounded to bf16
(round-to-nearest-even); targets y are uniform in [0, V_true).
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Tuple

import numpy as np

W_STD = 0.02
SEQ_LEN = 512
_CHUNK = 1 << 24  # elements per generation chunk (bounds temporary memory)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    V: int
    V_true: int
    seed: int = 0
    backward: bool = True
    g_kind: str = "normal"          # "normal" | "grpo"
    shards: Tuple[Tuple[int, int], ...] = ()   # (vocab_start, V_local) per shard; () = unsharded

    @property
    def flops_fwd(self) -> float:
        return 2.0 * self.T * self.H * self.V_true

    @property
    def flops_fwd_bwd(self) -> float:
        return 3.0 * self.flops_fwd

    def describe(self) -> dict:
        d = {"workload": self.name, "T": self.T, "H": self.H, "V": self.V, "V_true": self.V_true,
             "seed": self.seed, "backward": self.backward, "g": self.g_kind}
        if self.shards:
            d["shards"] = [list(s) for s in self.shards]
        return d


TINY = Workload("tiny", T=64, H=256, V=4096, V_true=4096, g_kind="normal")
QWEN3_8B_FWD = Workload("qwen3_8b_fwd", T=4096, H=4096, V=151936, V_true=151669, backward=False)
QWEN3_8B = Workload("qwen3_8b", T=8192, H=4096, V=151936, V_true=151669, g_kind="grpo")
QWEN3_30B_TP2 = Workload("qwen3_30b_tp2", T=16384, H=2048, V=151936, V_true=151669, g_kind="grpo",
                         shards=((0, 77824), (77824, 151936 - 77824)))
INVARIANCE_T = (1, 7, 128, 1000, 4097)
INVARIANCE_TARGETS = 128
INVARIANCE_H = 4096

CONFIGS: Dict[str, Workload] = {w.name: w for w in (TINY, QWEN3_8B_FWD, QWEN3_8B, QWEN3_30B_TP2)}


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest, ties to even. Inputs are finite."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    """bf16 bits of N(0, std^2) draws, generated in bounded chunks."""
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)
    for i in range(0, n, _CHUNK):
        k = min(_CHUNK, n - i)
        x = rng.standard_normal(k, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        out[i:i + k] = bf16_bits(x)
    return out.reshape(shape)


def _rng(seed: int, stream: int) -> np.random.Generator:
    # independent streams per tensor so that e.g. T does not change W
    return np.random.Generator(np.random.PCG64([seed, stream]))


def make_W(V: int, H: int, seed: int = 0) -> np.ndarray:
    return normal_bf16(_rng(seed, 1), (V, H), W_STD)


def make_h(T: int, H: int, seed: int = 0) -> np.ndarray:
    return normal_bf16(_rng(seed, 2), (T, H), 1.0)


def make_y(T: int, V_true: int, seed: int = 0) -> np.ndarray:
    return _rng(seed, 3).integers(0, V_true, size=T, dtype=np.int64)


def make_g(T: int, kind: str, seed: int = 0) -> np.ndarray:
    rng = _rng(seed, 4)
    if kind == "normal":
        return rng.standard_normal(T, dtype=np.float32)
    if kind == "grpo":
        n_seq = (T + SEQ_LEN - 1) // SEQ_LEN
        adv = rng.standard_normal(n_seq, dtype=np.float32)
        g = np.repeat(adv, SEQ_LEN)[:T] / np.float32(SEQ_LEN)
        return g.astype(np.float32)
    raise ValueError(kind)


def make_inputs(w: Workload, with_W: bool = True) -> Dict[str, np.ndarray]:
    """h (bf16 bits [T,H]), W (bf16 bits [V,H]), y (int64 [T]), g (float32 [T])."""
    d = {"h": make_h(w.T, w.H, w.seed), "y": make_y(w.T, w.V_true, w.seed),
         "g": make_g(w.T, w.g_kind, w.seed)}
    if with_W:
        d["W"] = make_W(w.V, w.H, w.seed)
    return d


def sparse_g(T: int, n_nonzero: int, seed: int = 0) -> Tuple[np.ndarray, np.ndarray]:
    """g with `n_nonzero` seeded non-zero N(0,1) entries at distinct positions; returns (g, positions)."""
    rng = _rng(seed, 5)
    pos = np.sort(rng.choice(T, size=min(n_nonzero, T), replace=False)).astype(np.int64)
    g = np.zeros(T, np.float32)
    g[pos] = rng.standard_normal(pos.shape[0], dtype=np.float32)
    return g, pos


def sample_rows(n_total: int, n: int, seed: int = 0, stream: int = 6) -> np.ndarray:
    """n distinct seeded indices in [0, n_total), always including the first and last."""
    rng = _rng(seed, stream)
    n = min(n, n_total)
    if n <= 2:
        return np.array(sorted({0, n_total - 1})[:n], dtype=np.int64)
    mid = rng.choice(np.arange(1, n_total - 1), size=n - 2, replace=False)
    return np.sort(np.concatenate([[0, n_total - 1], mid])).astype(np.int64)


@dataclasses.dataclass
class InvarianceBatch:
    T: int
    h: np.ndarray            # [T, H] bf16 bits
    y: np.ndarray            # [T]
    target_rows: np.ndarray  # [k] row of each embedded target inside this batch
    target_ids: np.ndarray   # [k] which of the 128 targets sits there


def invariance_targets(seed: int = 0, n: int = INVARIANCE_TARGETS, H: int = INVARIANCE_H,
                       V_true: int = 151669) -> Tuple[np.ndarray, np.ndarray]:
    """The fixed (hidden, target id) pairs whose logp must not depend on the batch."""
    rng = _rng(seed, 7)
    h = normal_bf16(rng, (n, H), 1.0)
    y = rng.integers(0, V_true, size=n, dtype=np.int64)
    return h, y


def invariance_batches(T: int, seed: int = 0, n: int = INVARIANCE_TARGETS, H: int = INVARIANCE_H,
                       V_true: int = 151669) -> List[InvarianceBatch]:
    """Ragged batches of size T holding all n targets at seeded positions among filler rows.

    T < n: the targets are spread over ceil(n/T) batches (a seeded permutation of
    all slots); T >= n: one batch holds them at distinct seeded rows.
    """
    th, ty = invariance_targets(seed, n, H, V_true)
    rng = _rng(seed + 1000 * T, 8)
    n_batches = (n + T - 1) // T
    slots = rng.permutation(n_batches * T)[:n]   # slot of target i
    out = []
    for b in range(n_batches):
        h = normal_bf16(rng, (T, H), 1.0)
        y = rng.integers(0, V_true, size=T, dtype=np.int64)
        ids = np.nonzero(slots // T == b)[0]
        rows = slots[ids] % T
        h[rows] = th[ids]
        y[rows] = ty[ids]
        out.append(InvarianceBatch(T, h, y, rows.astype(np.int64), ids.astype(np.int64)))
    return out
