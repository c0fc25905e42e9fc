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
    """q [B][Hq][Nq][D], k/v [B][Hkv][Nk][D] nested sequences of floats.

    The query rows are the last Nq positions of the Nk keys' sequence, so the
    causal mask lets row i see keys 0 .. i + Nk - Nq.
    Returns (o [B][Hq][Nq][D], lse [B][Hq][Nq]) as nested lists of floats."""
    B, Hq, Nq, D = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0])
    Hkv, Nk = len(k[0]), len(k[0][0])
    group = Hq // Hkv
    o = [[[[0.0] * D for _ in range(Nq)] for _ in range(Hq)] for _ in range(B)]
    lse = [[[0.0] * Nq for _ in range(Hq)] for _ in range(B)]
    for b in range(B):
        for h in range(Hq):
            hk = h // group
            for i in range(Nq):
                position = i + (Nk - Nq)  # of query row i within the key sequence
                allowed = [j for j in range(Nk) if not (causal and j > position)]
                w = {}
                for j in allowed:
                    dot = math.fsum(q[b][h][i][d] * k[b][hk][j][d] for d in range(D))
                    w[j] = math.exp(scale * dot)
                total = math.fsum(w.values())
                for d in range(D):
                    o[b][h][i][d] = math.fsum(w[j] * v[b][hk][j][d] for j in allowed) / total
                lse[b][h][i] = math.log(total)
    return o, lse
