"""Seeded synthetic inputs shared by the fp64 oracle and the CUDA path.

This module draws random numbers and lays out packed variable-length
batches.  It holds none of the attention arithmetic: it never computes a
score, a softmax statistic or a gradient.  Both the oracle tests and the
GPU tests call it, and neither side imports the other.

Recipe (all workloads are synthetic; the pages measure on no dataset):
  * Q, K, V, dO: float32 draws from N(0, 1) made by a CPU
    ``torch.Generator`` seeded with the case seed, then rounded to bf16
    (round-to-nearest-even, torch's conversion).  Each tensor uses its own
    sub-seed (seed*16 + index) so that adding a tensor never shifts another.
    Tensors of more than 2^31 elements are drawn the same way by a seeded
    generator on the device (bf16_normal_device).
  * Variable lengths: ``numpy.random.default_rng(seed).integers(lo, hi+1)``.
  * Packed layout ``[total, heads, head_dim]`` with cumulative int32
    offsets of B+1 entries, offsets[0] = 0 (the ``actual_q`` / ``actual_kv``
    arrays of the SK-16 single-pass FA Grad article, section 3).
  * Optional padding rows after the last sequence are filled with NaN so
    that a kernel reading them would leak NaN into its outputs.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


def bf16_normal(shape, seed: int, sub: int = 0) -> torch.Tensor:
    """N(0,1) float32 draws rounded to bf16, on the CPU."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) * 16 + int(sub))
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    return x.to(torch.bfloat16)


def bf16_normal_device(shape, seed: int, sub: int = 0, device="cuda", rows_per_draw: int = 1 << 16) -> torch.Tensor:
    """N(0,1) float32 draws rounded to bf16, drawn on the device by its own
    seeded generator (other values than bf16_normal for the same seed) in
    blocks of rows, for inputs too large to draw on the host."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 16 + int(sub))
    out = torch.empty(*shape, dtype=torch.bfloat16, device=device)
    for r0 in range(0, shape[0], rows_per_draw):
        r1 = min(shape[0], r0 + rows_per_draw)
        out[r0:r1] = torch.randn(r1 - r0, *shape[1:], generator=g, device=device, dtype=torch.float32)
    return out


def draw_lengths(n: int, lo: int, hi: int, seed: int) -> list[int]:
    """n integers uniform in [lo, hi] (inclusive)."""
    rng = np.random.default_rng(int(seed))
    return [int(x) for x in rng.integers(lo, hi + 1, size=n)]


def cumulative(lengths) -> np.ndarray:
    """B+1 cumulative offsets, int32, starting at 0."""
    cu = np.zeros(len(lengths) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    if cu[-1] > np.iinfo(np.int32).max:
        raise ValueError("total length does not fit int32 offsets")
    return cu.astype(np.int32)


@dataclasses.dataclass
class Case:
    """One attention-backward problem: shapes, mask and seed."""
    name: str
    heads: int
    head_dim: int
    q_lens: list
    kv_lens: list
    causal: bool
    seed: int
    pad_q: int = 0      # NaN rows appended after the last query row
    pad_kv: int = 0     # NaN rows appended after the last key row
    scale: float | None = None
    heads_kv: int | None = None   # key/value heads (grouped-query attention); None = heads
    window: int = 0               # causal sliding-window length (0 = none)
    bottom_right: bool = False    # causal diagonal aligned with the last key

    @property
    def batch(self) -> int:
        return len(self.q_lens)

    @property
    def kv_heads(self) -> int:
        return self.heads if self.heads_kv is None else self.heads_kv

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.head_dim)

    @property
    def cu_q(self) -> np.ndarray:
        return cumulative(self.q_lens)

    @property
    def cu_kv(self) -> np.ndarray:
        return cumulative(self.kv_lens)

    @property
    def total_q(self) -> int:
        return int(self.cu_q[-1]) + self.pad_q

    @property
    def total_kv(self) -> int:
        return int(self.cu_kv[-1]) + self.pad_kv

    def flops(self) -> float:
        """Algorithmic FLOPs of the backward: 10*s1*s2*d per head, halved
        under the causal mask (the counting rule of the target metric)."""
        tot = 0.0
        for s1, s2 in zip(self.q_lens, self.kv_lens):
            f = 10.0 * s1 * s2 * self.head_dim * self.heads
            tot += f / 2 if self.causal else f
        return tot

    def tensors(self):
        """Q, K, V, dO as CPU bf16 tensors, padding rows set to NaN."""
        H, Hkv, d = self.heads, self.kv_heads, self.head_dim
        q = bf16_normal((self.total_q, H, d), self.seed, 0)
        k = bf16_normal((self.total_kv, Hkv, d), self.seed, 1)
        v = bf16_normal((self.total_kv, Hkv, d), self.seed, 2)
        do = bf16_normal((self.total_q, H, d), self.seed, 3)
        nq, nkv = int(self.cu_q[-1]), int(self.cu_kv[-1])
        for t, n in ((q, nq), (do, nq), (k, nkv), (v, nkv)):
            t[n:] = float("nan")
        return q, k, v, do


def fixed(name, batch, heads, head_dim, s1, s2, causal, seed, **kw) -> Case:
    return Case(name, heads, head_dim, [s1] * batch, [s2] * batch, causal, seed, **kw)


# The five workloads of the target specification, seeds 1000 + k.
def cfg1() -> Case:
    return fixed("cfg1_tiny_b1_h1_d64_s128", 1, 1, 64, 128, 128, False, 1001)


def cfg2() -> Case:
    return fixed("cfg2_b2_h8_d128_s1024", 2, 8, 128, 1024, 1024, False, 1002)


def cfg3(causal: bool = True) -> Case:
    name = "cfg3_b4_h16_d128_s4096_" + ("causal" if causal else "noncausal")
    return fixed(name, 4, 16, 128, 4096, 4096, causal, 1003)


def cfg4() -> Case:
    lens = draw_lengths(8, 256, 8192, 1004)
    return Case("cfg4_varlen8_h32_d128_causal", 32, 128, lens, list(lens), True, 1004)


def cfg5() -> Case:
    ql = draw_lengths(4, 512, 2048, 1005)
    kl = draw_lengths(4, 2048, 8192, 2005)
    return Case("cfg5_cross4_h16_d64", 16, 64, ql, kl, False, 1005)


CONFIGS = {"cfg1": cfg1, "cfg2": cfg2, "cfg3": lambda: cfg3(True),
           "cfg3nc": lambda: cfg3(False), "cfg4": cfg4, "cfg5": cfg5}


# Workloads of the variants (grouped-query attention, masks): shapes of the
# common uses, seeds 1100 + k.
def gqa() -> Case:
    """32 query heads sharing 8 key/value heads, causal, 4 x 4096 tokens."""
    return fixed("gqa_b4_h32_hkv8_s4096_d128_causal", 4, 32, 128, 4096, 4096, True, 1101, heads_kv=8)


def swa() -> Case:
    """Causal sliding window of 4096 keys over 2 x 16384 tokens."""
    return fixed("swa_b2_h16_s16384_w4096_d128", 2, 16, 128, 16384, 16384, True, 1102, window=4096)


def br() -> Case:
    """Bottom-right causal: 1024 new queries against 8192 keys (the last
    1024 of them the queries' own), 8 sequences."""
    return fixed("br_b8_h16_s1024_s8192_d128", 8, 16, 128, 1024, 8192, True, 1103, bottom_right=True)


def d256(causal: bool = False) -> Case:
    """head_dim 256, 4 x 4096 tokens, 8 heads (the FLOPs of cfg3)."""
    name = "d256_b4_h8_s4096_" + ("causal" if causal else "noncausal")
    return fixed(name, 4, 8, 256, 4096, 4096, causal, 1104)


VARIANTS = {"gqa": gqa, "swa": swa, "br": br, "d256": lambda: d256(False), "d256c": lambda: d256(True)}
