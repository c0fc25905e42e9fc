"""Pins for the float64 attention oracle.

Each pin checks an oracle callable ``att(q, k, v, scale, causal) -> (o, lse)``
against a fact that does not come from the oracle itself: a closed form, an
invariant of the mathematics, an independent library routine (scipy's softmax
and logsumexp, torch's scaled_dot_product_attention in float64) or a brute-force
triple loop.  A pin raises AssertionError when the oracle breaks it.

The facts follow the definition on the page "从零开始写Qwen3"
(deepseek.csdn.net/6a3201f8..., sections "简易情况-三矩阵相乘" and
"FlashAttention"): O = softmax(mask(Q K^T * scale)) V with the causal mask
j <= i and kv_head = q_head // (Hq / Hkv); LSE is the natural-log
log-sum-exp of the masked, scaled score row.
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import logsumexp, softmax

TOL = 1e-12


def _close(a, b, tol=TOL, what=""):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    err = np.max(np.abs(a - b) / np.maximum(1.0, np.abs(b))) if a.size else 0.0
    assert err <= tol, f"{what}: max rel err {err:.3e} > {tol:.1e}"


def _rand(rng, *shape, std=1.0):
    return rng.standard_normal(shape) * std


def _scores(q, k, scale, causal):
    """Independent masked score tensor [B,Hq,N,N] (numpy einsum, contiguous groups)."""
    B, Hq, N, D = q.shape
    G = Hq // k.shape[1]
    kk = np.repeat(k, G, axis=1)  # head h reads kv head h // G
    s = scale * np.einsum("bhid,bhjd->bhij", q, kk)
    if causal:
        s = np.where(np.tril(np.ones((N, N), dtype=bool)), s, -np.inf)
    return s


def pin_zero_query(att):
    """Q = 0: every allowed logit is 0, so O_i is the mean of the allowed V rows and
    LSE_i = ln(#allowed) -- prefix means for the causal mask."""
    rng = np.random.default_rng(1)
    B, Hq, Hkv, N, D = 2, 4, 2, 37, 8
    q = np.zeros((B, Hq, N, D))
    k = _rand(rng, B, Hkv, N, D)
    v = _rand(rng, B, Hkv, N, D)
    for causal in (True, False):
        o, lse = att(q, k, v, 0.3, causal)
        for h in range(Hq):
            vh = v[:, h // 2]
            if causal:
                want = np.cumsum(vh, axis=1) / np.arange(1, N + 1)[None, :, None]
                want_lse = np.log(np.arange(1, N + 1))[None, :].repeat(B, 0)
            else:
                want = np.repeat(vh.mean(axis=1, keepdims=True), N, axis=1)
                want_lse = np.full((B, N), math.log(N))
            _close(o[:, h], want, what=f"zero-Q O causal={causal} h={h}")
            _close(lse[:, h], want_lse, what=f"zero-Q LSE causal={causal} h={h}")


def pin_identity_values(att):
    """V = identity (N <= D): O_i is the attention-weight row itself.  Its entries are
    exp(s_ij - LSE_i) with s from an independent einsum, zero above the diagonal
    under the causal mask, and they sum to 1."""
    rng = np.random.default_rng(2)
    B, Hq, Hkv, N, D = 1, 4, 2, 12, 16
    q = _rand(rng, B, Hq, N, D)
    k = _rand(rng, B, Hkv, N, D)
    v = np.zeros((B, Hkv, N, D))
    v[:, :, np.arange(N), np.arange(N)] = 1.0
    scale = 0.37
    for causal in (True, False):
        o, lse = att(q, k, v, scale, causal)
        s = _scores(q, k, scale, causal)
        w = np.exp(s - lse[..., None])
        _close(o[..., :N], w, what=f"weights causal={causal}")
        _close(o[..., N:], np.zeros_like(o[..., N:]), what="weights padding")
        _close(o.sum(-1), np.ones((B, Hq, N)), what=f"row sums causal={causal}")
        if causal:
            assert np.all(o[..., :N][..., ~np.tril(np.ones((N, N), dtype=bool))] == 0.0), \
                "weight above the diagonal"


def pin_library_softmax(att):
    """General inputs against scipy: O = softmax(S) V and LSE = logsumexp(S) over the
    masked, scaled scores; large logits (std ~ 16) stress the max shift."""
    rng = np.random.default_rng(3)
    B, Hq, Hkv, N, D = 2, 6, 3, 45, 16
    q = _rand(rng, B, Hq, N, D, std=4.0)
    k = _rand(rng, B, Hkv, N, D, std=4.0)
    v = _rand(rng, B, Hkv, N, D)
    for causal in (True, False):
        o, lse = att(q, k, v, 1.0 / math.sqrt(D), causal)
        s = _scores(q, k, 1.0 / math.sqrt(D), causal)
        p = softmax(s, axis=-1)
        want = np.einsum("bhij,bhjd->bhid", p, np.repeat(v, Hq // Hkv, axis=1))
        _close(o, want, tol=1e-11, what=f"softmax·V causal={causal}")
        _close(lse, logsumexp(s, axis=-1), what=f"logsumexp causal={causal}")


def pin_selection(att):
    """One logit per row dominates by 1000: O_i is exactly that V row and LSE_i is
    that logit.  Under the causal mask a row whose dominant key lies in the future
    sees only zero logits and takes the prefix mean."""
    rng = np.random.default_rng(4)
    B, Hq, Hkv, N, D = 1, 1, 1, 16, 16
    perm = rng.permutation(N)
    q = np.zeros((B, Hq, N, D))
    q[0, 0, np.arange(N), np.arange(N)] = 1.0
    k = np.zeros((B, Hkv, N, D))
    k[0, 0, np.arange(N), perm] = 1.0  # key j points at query row perm[j]
    v = _rand(rng, B, Hkv, N, D)
    scale = 1000.0
    inv = np.argsort(perm)  # row i's dominant key
    for causal in (False, True):
        o, lse = att(q, k, v, scale, causal)
        for i in range(N):
            j = inv[i]
            if causal and j > i:
                _close(o[0, 0, i], v[0, 0, : i + 1].mean(0), what=f"row {i} masked winner")
                _close(lse[0, 0, i], math.log(i + 1), what=f"row {i} LSE masked winner")
            else:
                assert np.array_equal(o[0, 0, i], v[0, 0, j]), f"row {i} not V[{j}]"
                assert lse[0, 0, i] == scale, f"row {i} LSE {lse[0, 0, i]} != {scale}"


def pin_shift(att):
    """Adding one vector u to every key row adds scale*<q_i,u> to every logit of row i:
    O is unchanged and LSE moves by exactly that amount."""
    rng = np.random.default_rng(5)
    B, Hq, Hkv, N, D = 1, 4, 1, 33, 8
    q = _rand(rng, B, Hq, N, D)
    k = _rand(rng, B, Hkv, N, D)
    v = _rand(rng, B, Hkv, N, D)
    u = _rand(rng, D, std=2.0)
    scale = 0.5
    for causal in (True, False):
        o1, l1 = att(q, k, v, scale, causal)
        o2, l2 = att(q, k + u, v, scale, causal)
        _close(o2, o1, tol=1e-11, what="shift O")
        _close(l2, l1 + scale * np.einsum("bhid,d->bhi", q, u), tol=1e-11, what="shift LSE")


def pin_gqa_vs_mha(att):
    """Grouped heads equal multi-head attention on K, V repeated G times along the head
    axis with contiguous groups (q heads gG..gG+G-1 read kv head g)."""
    rng = np.random.default_rng(6)
    B, Hq, Hkv, N, D = 2, 6, 2, 20, 8
    q = _rand(rng, B, Hq, N, D)
    k = _rand(rng, B, Hkv, N, D)
    v = _rand(rng, B, Hkv, N, D)
    for causal in (True, False):
        o1, l1 = att(q, k, v, 0.4, causal)
        o2, l2 = att(q, np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1), 0.4, causal)
        _close(o1, o2, what="GQA vs MHA O")
        _close(l1, l2, what="GQA vs MHA LSE")


def pin_permutation(att):
    """Without the mask, permuting the key/value rows jointly changes nothing."""
    rng = np.random.default_rng(7)
    B, Hq, Hkv, N, D = 1, 2, 1, 29, 8
    q = _rand(rng, B, Hq, N, D)
    k = _rand(rng, B, Hkv, N, D)
    v = _rand(rng, B, Hkv, N, D)
    perm = rng.permutation(N)
    o1, l1 = att(q, k, v, 0.6, False)
    o2, l2 = att(q, k[:, :, perm], v[:, :, perm], 0.6, False)
    _close(o1, o2, tol=1e-11, what="permutation O")
    _close(l1, l2, tol=1e-11, what="permutation LSE")


def pin_single_key(att):
    """N = 1: the only weight is 1, so O = V[0] and LSE = scale*<q, k_0>."""
    rng = np.random.default_rng(8)
    q = _rand(rng, 2, 4, 1, 8)
    k = _rand(rng, 2, 2, 1, 8)
    v = _rand(rng, 2, 2, 1, 8)
    for causal in (True, False):
        o, lse = att(q, k, v, 0.7, causal)
        _close(o, np.repeat(v, 2, axis=1), what="N=1 O")
        _close(lse, 0.7 * np.einsum("bhid,bhid->bhi", q, np.repeat(k, 2, axis=1)), what="N=1 LSE")


def pin_causality(att):
    """Under the causal mask, rows j > i of K and V never reach output row i."""
    rng = np.random.default_rng(9)
    B, Hq, Hkv, N, D = 1, 2, 1, 24, 8
    q = _rand(rng, B, Hq, N, D)
    k = _rand(rng, B, Hkv, N, D)
    v = _rand(rng, B, Hkv, N, D)
    o1, l1 = att(q, k, v, 0.5, True)
    cut = 10
    k2, v2 = k.copy(), v.copy()
    k2[:, :, cut + 1:] = _rand(rng, B, Hkv, N - cut - 1, D, std=10.0)
    v2[:, :, cut + 1:] = _rand(rng, B, Hkv, N - cut - 1, D, std=10.0)
    o2, l2 = att(q, k2, v2, 0.5, True)
    assert np.array_equal(o1[:, :, : cut + 1], o2[:, :, : cut + 1]), "future rows leaked"
    assert np.array_equal(l1[:, :, : cut + 1], l2[:, :, : cut + 1]), "future rows leaked (LSE)"


def pin_naive(att):
    """Tiny inputs against the pure-Python triple loop (textbook softmax, fsum)."""
    from oracle.naive import attention_naive

    rng = np.random.default_rng(10)
    B, Hq, Hkv, N, D = 1, 2, 1, 7, 5
    q = _rand(rng, B, Hq, N, D)
    k = _rand(rng, B, Hkv, N, D)
    v = _rand(rng, B, Hkv, N, D)
    for causal in (True, False):
        o, lse = att(q, k, v, 0.45, causal)
        on, ln = attention_naive(q.tolist(), k.tolist(), v.tolist(), 0.45, causal)
        _close(o, np.array(on), what=f"naive O causal={causal}")
        _close(lse, np.array(ln), what=f"naive LSE causal={causal}")


def pin_torch_sdpa(att):
    """Against torch's scaled_dot_product_attention in float64 on the CPU (heads expanded
    contiguously; its is_causal mask is the top-left j <= i mask for square inputs)."""
    import torch

    rng = np.random.default_rng(11)
    B, Hq, Hkv, N, D = 2, 8, 2, 50, 32
    q = _rand(rng, B, Hq, N, D)
    k = _rand(rng, B, Hkv, N, D)
    v = _rand(rng, B, Hkv, N, D)
    scale = 1.0 / math.sqrt(D)
    for causal in (True, False):
        o, _ = att(q, k, v, scale, causal)
        t = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q), torch.from_numpy(np.repeat(k, 4, axis=1)),
            torch.from_numpy(np.repeat(v, 4, axis=1)), is_causal=causal, scale=scale)
        _close(o, t.numpy(), tol=1e-11, what=f"torch sdpa causal={causal}")


# ------------------------------------------------------------------ Nq != Nk
# A block of Nq query rows attending over Nk >= Nq keys: the queries are the last
# Nq positions of the keys' sequence, so the causal mask is aligned at the bottom
# right (row i sees keys j <= i + Nk - Nq).


def _mask_bottom_right(nq, nk):
    return np.tril(np.ones((nq, nk), dtype=bool), k=nk - nq)


def pin_bottom_right_library(att):
    """Nq < Nk against scipy softmax / logsumexp over an explicitly built
    bottom-right mask; Nq = 1 (one new token) sees every key."""
    rng = np.random.default_rng(12)
    B, Hq, Hkv, D = 2, 4, 2, 16
    for nq, nk in ((1, 45), (7, 45), (30, 31), (13, 200)):
        q = _rand(rng, B, Hq, nq, D, std=2.0)
        k = _rand(rng, B, Hkv, nk, D, std=2.0)
        v = _rand(rng, B, Hkv, nk, D)
        for causal in (True, False):
            o, lse = att(q, k, v, 0.25, causal)
            kk, vv = np.repeat(k, Hq // Hkv, axis=1), np.repeat(v, Hq // Hkv, axis=1)
            s = 0.25 * np.einsum("bhid,bhjd->bhij", q, kk)
            if causal:
                s = np.where(_mask_bottom_right(nq, nk), s, -np.inf)
            want = np.einsum("bhij,bhjd->bhid", softmax(s, axis=-1), vv)
            _close(o, want, tol=1e-11, what=f"Nq={nq} Nk={nk} causal={causal} O")
            _close(lse, logsumexp(s, axis=-1), what=f"Nq={nq} Nk={nk} causal={causal} LSE")


def pin_chunk_suffix(att):
    """A causal query block equals the last Nq rows of the square causal problem whose
    queries are a prefix followed by that block (chunked prefill)."""
    rng = np.random.default_rng(13)
    B, Hq, Hkv, D = 1, 6, 2, 8
    for nq, nk in ((5, 40), (17, 17 + 128), (1, 9)):
        q_tail = _rand(rng, B, Hq, nq, D)
        q_full = np.concatenate([_rand(rng, B, Hq, nk - nq, D), q_tail], axis=2)
        k = _rand(rng, B, Hkv, nk, D)
        v = _rand(rng, B, Hkv, nk, D)
        o1, l1 = att(q_tail, k, v, 0.5, True)
        o2, l2 = att(q_full, k, v, 0.5, True)
        _close(o1, o2[:, :, nk - nq:], what=f"suffix O Nq={nq} Nk={nk}")
        _close(l1, l2[:, :, nk - nq:], what=f"suffix LSE Nq={nq} Nk={nk}")


def pin_naive_nonsquare(att):
    """Tiny Nq < Nk inputs against the pure-Python triple loop."""
    from oracle.naive import attention_naive

    rng = np.random.default_rng(14)
    q = _rand(rng, 1, 2, 3, 4)
    k = _rand(rng, 1, 1, 8, 4)
    v = _rand(rng, 1, 1, 8, 4)
    for causal in (True, False):
        o, lse = att(q, k, v, 0.6, causal)
        on, ln = attention_naive(q.tolist(), k.tolist(), v.tolist(), 0.6, causal)
        _close(o, np.array(on), what=f"naive Nq<Nk O causal={causal}")
        _close(lse, np.array(ln), what=f"naive Nq<Nk LSE causal={causal}")


def pin_torch_sdpa_nonsquare(att):
    """torch float64 scaled_dot_product_attention with the bottom-right mask passed
    as an explicit boolean attn_mask (its is_causal is top-left for Nq != Nk)."""
    import torch

    rng = np.random.default_rng(15)
    B, Hq, Hkv, nq, nk, D = 2, 8, 2, 19, 77, 32
    q = _rand(rng, B, Hq, nq, D)
    k = _rand(rng, B, Hkv, nk, D)
    v = _rand(rng, B, Hkv, nk, D)
    scale = 1.0 / math.sqrt(D)
    o, _ = att(q, k, v, scale, True)
    t = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(np.repeat(k, 4, axis=1)),
        torch.from_numpy(np.repeat(v, 4, axis=1)),
        attn_mask=torch.from_numpy(_mask_bottom_right(nq, nk)), scale=scale)
    _close(o, t.numpy(), tol=1e-11, what="torch sdpa bottom-right")


ALL_PINS = [pin_zero_query, pin_identity_values, pin_library_softmax, pin_selection,
            pin_shift, pin_gqa_vs_mha, pin_permutation, pin_single_key, pin_causality,
            pin_naive, pin_torch_sdpa, pin_bottom_right_library, pin_chunk_suffix,
            pin_naive_nonsquare, pin_torch_sdpa_nonsquare]
