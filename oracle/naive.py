"""Pure-Python triple loop for tiny attention inputs (TEST INFRASTRUCTURE ONLY).

The textbook softmax without the max shift, with exactly rounded sums
(``math.fsum``), so its rounding differs from the C oracle's sequential sums.
It follows the softmax form of O on the page "从零开始写Qwen3"
(deepseek.csdn.net/6a3201f8..., section "简易情况-三矩阵相乘") and the causal
mask and kv-head grouping of its section "FlashAttention".  Use it only where
exp(score) neither overflows nor underflows (tiny inputs, moderate logits).
"""
from __future__ import annotations

import math


def attention_naive(q, k, v, scale, causal):
    """q [B][Hq][N][D], k/v [B][Hkv][N][D] nested sequences of floats.

    Returns (o [B][Hq][N][D], lse [B][Hq][N]) as nested lists of floats."""
    B, Hq, N, D = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0])
    Hkv = len(k[0])
    group = Hq // Hkv
    o = [[[[0.0] * D for _ in range(N)] for _ in range(Hq)] for _ in range(B)]
    lse = [[[0.0] * N for _ in range(Hq)] for _ in range(B)]
    for b in range(B):
        for h in range(Hq):
            hk = h // group
            for i in range(N):
                allowed = [j for j in range(N) if not (causal and j > i)]
                w = {}
                for j in allowed:
                    dot = math.fsum(q[b][h][i][d] * k[b][hk][j][d] for d in range(D))
                    w[j] = math.exp(scale * dot)
                total = math.fsum(w.values())
                for d in range(D):
                    o[b][h][i][d] = math.fsum(w[j] * v[b][hk][j][d] for j in allowed) / total
                lse[b][h][i] = math.log(total)
    return o, lse
