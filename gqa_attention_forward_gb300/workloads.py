"""Seeded synthetic inputs for the fused GQA attention forward pass.

This module serves both the CUDA path and the float64 oracle, so it holds no
attention arithmetic: only the workload table, random draws from a seeded
generator, and rounding of the draws to the 16-bit storage type.  Inputs are
returned as uint16 storage words; each side decodes them on its own.

The workloads follow the shapes and value distributions of the pages'
benchmarks: the Triton tuning page "从零开始写Qwen3" (deepseek.csdn.net/6a31faef...,
section "基准": B=2, N=1024, H=16/8, D=128, float16) and the grouped-query
prefill setting of the derivation page "从零开始写Qwen3" (deepseek.csdn.net/
6a3201f8..., section "概述": prefill over a prompt of length S).  Every value
is i.i.d. normal; the tail/stress workload widens Q and K to std 4 so that
logits have std 16 and rows are close to one-hot.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    N: int
    D: int
    dtype: str  # "f16" or "bf16"
    causal: bool
    q_std: float = 1.0
    k_std: float = 1.0
    v_std: float = 1.0
    seed: int = 1234
    Nk: int | None = None  # keys per head when it differs from the N query rows
    entry: str = "attn_fwd"  # C entry point: "attn_fwd", "attn_fwd_decode" or "attn_fwd_kv_split"

    @property
    def n_keys(self) -> int:
        return self.N if self.Nk is None else self.Nk

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def flops(self) -> float:
        """Counted FLOPs: 4*B*Hq*N*Nk*D; with the causal mask the query block
        drops the upper triangle of its last N columns: 4*B*Hq*D*(N*Nk - N^2/2),
        which is 2*B*Hq*N^2*D for N == Nk."""
        n, nk = float(self.N), float(self.n_keys)
        pairs = n * nk - n * n / 2.0 if self.causal else n * nk
        return 4.0 * self.B * self.Hq * self.D * pairs

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_causal_gqa_f16", 1, 2, 1, 128, 64, "f16", True, seed=1234),
        Workload("pages_shape_causal_gqa_f16", 2, 16, 8, 1024, 128, "f16", True, seed=1235),
        Workload("noncausal_gqa_bf16_n4096", 4, 32, 8, 4096, 128, "bf16", False, seed=1236),
        Workload("long_prefill_causal_gqa_bf16_n32768", 1, 32, 8, 32768, 128, "bf16", True,
                 seed=1237),
        Workload("tail_stress_causal_gqa_bf16_n2000", 8, 64, 8, 2000, 128, "bf16", True,
                 q_std=4.0, k_std=4.0, v_std=1.0, seed=1238),
        # a 4096-token chunk of the long prefill over its 32768 keys (bottom-right mask)
        Workload("chunked_prefill_causal_gqa_bf16_q4096_k32768", 1, 32, 8, 4096, 128, "bf16",
                 True, seed=1239, Nk=32768),
        # one new token over the long prefill's keys, and a batch of such steps:
        # grouped-query packing and key splits (attn_fwd_decode)
        Workload("decode_gqa_bf16_b1_q1_k32768", 1, 32, 8, 1, 128, "bf16", True, seed=1240,
                 Nk=32768, entry="attn_fwd_decode"),
        Workload("decode_gqa_bf16_b16_q1_k8192", 16, 32, 8, 1, 128, "bf16", True, seed=1241,
                 Nk=8192, entry="attn_fwd_decode"),
        Workload("short_chunk_gqa_bf16_q16_k32768", 1, 32, 8, 16, 128, "bf16", True, seed=1242,
                 Nk=32768, entry="attn_fwd_decode"),
        # the equal-length workloads through attn_fwd_kv_split (last round cut along the
        # keys); same shapes and inputs as their plain entries above
        Workload("noncausal_gqa_bf16_n4096_split", 4, 32, 8, 4096, 128, "bf16", False, seed=1236,
                 entry="attn_fwd_kv_split"),
        Workload("chunked_prefill_causal_gqa_bf16_q4096_k32768_split", 1, 32, 8, 4096, 128, "bf16",
                 True, seed=1239, Nk=32768, entry="attn_fwd_kv_split"),
    ]
}
ORDER = list(WORKLOADS)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even) as uint16 words."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to IEEE half (nearest, ties to even) as uint16 words."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    if dtype == "f16":
        return f32_to_f16_bits(x)
    raise ValueError(f"unknown dtype {dtype!r}")


def make_inputs(w: Workload, seed: int | None = None):
    """q [B,Hq,N,D], k and v [B,Hkv,Nk,D] as uint16 storage words of w.dtype.

    Draw order is q, k, v from one numpy PCG64 generator seeded with w.seed."""
    rng = np.random.default_rng(w.seed if seed is None else seed)
    out = {}
    for name, heads, rows, std in (("q", w.Hq, w.N, w.q_std), ("k", w.Hkv, w.n_keys, w.k_std),
                                   ("v", w.Hkv, w.n_keys, w.v_std)):
        x = rng.standard_normal((w.B, heads, rows, w.D), dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        out[name] = to_bits(x, w.dtype)
    return out


def sample_rows(w: Workload, count: int, seed: int = 99) -> np.ndarray:
    """Flattened (b*Hq + hq)*N + i indices of a stratified row sample.

    Covers the first and last rows, the rows on both sides of every 128-row
    boundary the sample reaches, and random rows across all heads."""
    rng = np.random.default_rng(seed)
    BH, N = w.B * w.Hq, w.N
    special = {0, 1, N - 1, N - 2, min(127, N - 1), min(128, N - 1), min(129, N - 1),
               max(0, N - 129), (N // 128) * 128 - 1 if N >= 128 else 0}
    picks = []
    for bh in range(BH):
        for i in sorted(special):
            if 0 <= i < N:
                picks.append(bh * N + i)
    picks = sorted(set(picks))
    if len(picks) > count // 2:
        picks = list(rng.choice(np.array(picks), count // 2, replace=False))
    rest = count - len(picks)
    if rest > 0:
        picks.extend(rng.integers(0, BH * N, size=rest).tolist())
    return np.array(sorted(set(int(p) for p in picks)), dtype=np.int64)
