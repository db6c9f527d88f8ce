"""Seeded synthetic workloads for causal packed attention (inputs only).

This module is the one piece shared by the oracle side and the CUDA side: it
draws the bf16 inputs and the document lengths.  It holds none of the
method's arithmetic (no quantizer, no attention, no codec).

Workload shapes follow the packed causal training-call workloads of the FLAMIA
paper (Table 1 of "FLAMIA: FLAsh MIcroscaling Attention", as summarised in the
FLAMIA technical review, section 8 "Time the training call"): documents packed
into one row through cu_seqlens, 16-32 query heads, head dim 64 or 128.

Draw order from ``numpy.random.default_rng(seed)``: document lengths (when the
workload draws them), then Q, K, V, dO, each a float32 array of shape
``[T, H, d]`` rounded to bf16 with round-to-nearest-even.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    lengths: tuple            # document lengths, in packed order
    hq: int
    hkv: int
    d: int
    dist: str = "normal"      # "normal" | "student_t3" | "normal_outliers"
    seed: int = 0
    description: str = ""
    # visible keys: query i sees key j of its document iff i - left <= j <= i + right
    # (-1: no limit); causal (-1, 0), noncausal (-1, -1)
    window: tuple = (-1, 0)

    @property
    def causal(self) -> bool:
        return self.window[1] == 0

    @property
    def total_tokens(self) -> int:
        return int(sum(self.lengths))

    @property
    def cu_seqlens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.lengths)]).astype(np.int32)


def packed_lengths(total: int, lo: int, hi: int, seed: int) -> List[int]:
    """Draw lengths uniformly in [lo, hi] until they reach ``total`` tokens;
    the last document is truncated to the remainder (it may be shorter than lo)."""
    rng = np.random.default_rng(seed)
    out, acc = [], 0
    while acc < total:
        n = int(rng.integers(lo, hi + 1))
        n = min(n, total - acc)
        out.append(n)
        acc += n
    return out


def _workloads():
    w = {}
    w["causal_b1_h2_s256_d64"] = Workload(
        "causal_b1_h2_s256_d64", (256,), 2, 2, 64,
        description="single causal batched call, B=1, H=2, seq 256, d=64")
    w["packed_16k_h16_d128"] = Workload(
        "packed_16k_h16_d128", tuple(packed_lengths(16384, 128, 4096, 0)), 16, 16, 128,
        description="packed varlen MHA, 16384 tokens, lengths U[128,4096], H=16, d=128")
    w["gqa_b4_s8192_hq32_hkv8_d128"] = Workload(
        "gqa_b4_s8192_hq32_hkv8_d128", (8192,) * 4, 32, 8, 128,
        description="GQA causal batched, B=4, seq 8192, 32 query / 8 kv heads, d=128")
    w["mixed_nvfp4_gqa_b4_s8192"] = Workload(
        "mixed_nvfp4_gqa_b4_s8192", (8192,) * 4, 32, 8, 128, dist="normal_outliers",
        description="GQA shape with 0.1% outliers x100 (mixed NVFP4 score path)")
    w["strict_packed_4x8192_h16_t3"] = Workload(
        "strict_packed_4x8192_h16_t3", (8192,) * 4, 16, 16, 128, dist="student_t3",
        description="4 documents of 8192, H=16, d=128, Student-t(3) inputs, strict options")
    # the skewed packed row of the pages' training-call table: one long document and many
    # short ones (the layout where the cost-ordered work list matters most)
    w["skewed_8192_224x256_h16_d128"] = Workload(
        "skewed_8192_224x256_h16_d128", (8192,) + (256,) * 224, 16, 16, 128,
        description="packed causal MHA, one 8192-token document and 224 of 256 tokens, H=16, d=128")
    # the uniform packed row of the same table: sixteen documents of 4096 tokens
    w["packed_16x4096_h16_d128"] = Workload(
        "packed_16x4096_h16_d128", (4096,) * 16, 16, 16, 128,
        description="packed causal MHA, 16 documents of 4096 tokens, H=16, d=128")
    # the noncausal calls the pages time beside the causal ones (packed rows, and the
    # batched 2 x 8192 case)
    w["noncausal_packed_16k_h16_d128"] = Workload(
        "noncausal_packed_16k_h16_d128", tuple(packed_lengths(16384, 128, 4096, 0)), 16, 16, 128,
        window=(-1, -1), description="packed varlen MHA as packed_16k_h16_d128, noncausal")
    w["noncausal_b2_s8192_h16_d128"] = Workload(
        "noncausal_b2_s8192_h16_d128", (8192,) * 2, 16, 16, 128, window=(-1, -1),
        description="batched noncausal, B=2, seq 8192, H=16, d=128")
    return w


WORKLOADS = _workloads()


def custom(lengths, hq, hkv, d, dist="normal", seed=0, name="custom", window=(-1, 0)) -> Workload:
    return Workload(name, tuple(int(x) for x in lengths), int(hq), int(hkv), int(d), dist, int(seed),
                    window=tuple(window))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); return the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def _draw(rng, shape, dist):
    if dist == "normal":
        return rng.standard_normal(shape, dtype=np.float32)
    if dist == "student_t3":
        return rng.standard_t(3, size=shape).astype(np.float32)
    if dist == "normal_outliers":
        x = rng.standard_normal(shape, dtype=np.float32)
        n = x.size
        k = max(1, n // 1000)
        idx = rng.choice(n, size=k, replace=False)
        x.reshape(-1)[idx] *= 100.0
        return x
    raise ValueError(dist)


def make_inputs(w: Workload, seed: Optional[int] = None, tensors=("q", "k", "v", "do")):
    """Return dict of bf16 bit arrays (uint16) with shapes q/do [T,hq,d], k/v [T,hkv,d]."""
    rng = np.random.default_rng(w.seed if seed is None else seed)
    T = w.total_tokens
    shapes = {"q": (T, w.hq, w.d), "k": (T, w.hkv, w.d), "v": (T, w.hkv, w.d), "do": (T, w.hq, w.d)}
    out = {}
    for name in ("q", "k", "v", "do"):
        x = _draw(rng, shapes[name], w.dist)
        if name in tensors:
            out[name] = f32_to_bf16_bits(x)
    return out


def visible_pair_count(lengths, window=(-1, 0)) -> int:
    """Number of (query, key) pairs the mask admits (the FLOP count's unit):
    sum n(n+1)/2 for causal calls, sum n^2 for noncausal ones, and for a window
    (left, right) the sum over rows i of |[max(0, i - left), min(n - 1, i + right)]|."""
    left, right = window
    if left < 0 and right == 0:
        return int(sum(int(n) * (int(n) + 1) // 2 for n in lengths))
    total = 0
    for n in lengths:
        i = np.arange(int(n), dtype=np.int64)
        lo = np.zeros_like(i) if left < 0 else np.maximum(i - left, 0)
        hi = np.full_like(i, int(n) - 1) if right < 0 else np.minimum(i + right, int(n) - 1)
        total += int((hi - lo + 1).sum())
    return total
