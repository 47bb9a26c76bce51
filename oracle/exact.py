"""Exact fp64 softmax attention on packed documents, forward and backward.

Source: "FLAMIA: FLAsh MIcroscaling Attention ..." Section 2, "FlashAttention"
paragraph: S = Q K^T / sqrt(d), P = softmax(S), O = P V; backward
dV = P^T dO, dP = dO V^T, dS = P o (dP - D) with D_i = sum_j P_ij dP_ij
(= dO_i . O_i), dQ = dS K, dK = dS^T Q (the 1/sqrt(d) of S carried into dQ
and dK).  Section 3.6.1: documents packed in one row attend only within
themselves; rows outside every document get LSE = +inf and zero output.
Grouped-query heads: query head h reads key/value head h // (Hq / Hkv), and
dK, dV sum over the query heads of a group.

Pinned by tests/test_oracle_exact.py against textbook per-document softmax,
torch scaled_dot_product_attention in float64 with a block-diagonal causal
mask, central finite differences of <dO, O>, and the identities
D = sum_j P o dP and sum_j dS_ij = 0.
"""
from __future__ import annotations

import numpy as np


def _doc_ranges(cu_seqlens):
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    return [(int(cu[r]), int(cu[r + 1])) for r in range(len(cu) - 1)]


def _probs(q_h, k_h, causal):
    d = q_h.shape[-1]
    S = (q_h @ k_h.T) / np.sqrt(d)
    if causal:
        L = S.shape[0]
        S = np.where(np.tril(np.ones((L, L), dtype=bool)), S, -np.inf)
    m = S.max(axis=1, keepdims=True)
    e = np.exp(S - m)
    l = e.sum(axis=1, keepdims=True)
    return e / l, (m + np.log(l))[:, 0]


def forward(q, k, v, cu_seqlens, causal: bool = True, heads=None):
    """O [T, Hq, d] and LSE [Hq, T] (natural log) for the query heads in ``heads`` (default: all)."""
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64); v = np.asarray(v, np.float64)
    T, Hq, d = q.shape
    g = Hq // k.shape[1]
    heads = range(Hq) if heads is None else heads
    O = np.zeros((T, Hq, d))
    lse = np.full((Hq, T), np.inf)
    for s, e in _doc_ranges(cu_seqlens):
        if e <= s:
            continue
        for h in heads:
            P, lse_h = _probs(q[s:e, h], k[s:e, h // g], causal)
            O[s:e, h] = P @ v[s:e, h // g]
            lse[h, s:e] = lse_h
    return O, lse


def backward(q, k, v, do, cu_seqlens, causal: bool = True, heads=None):
    """dQ [T, Hq, d], dK, dV [T, Hkv, d] (sums over the query heads in ``heads``)."""
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64); do = np.asarray(do, np.float64)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    heads = range(Hq) if heads is None else heads
    dq = np.zeros_like(q); dk = np.zeros_like(k); dv = np.zeros_like(v)
    for s, e in _doc_ranges(cu_seqlens):
        if e <= s:
            continue
        for h in heads:
            hk = h // g
            P, _ = _probs(q[s:e, h], k[s:e, hk], causal)
            O = P @ v[s:e, hk]
            dP = do[s:e, h] @ v[s:e, hk].T
            D = (do[s:e, h] * O).sum(axis=1)
            dS = P * (dP - D[:, None])
            dq[s:e, h] = dS @ k[s:e, hk] / np.sqrt(d)
            dk[s:e, hk] += dS.T @ q[s:e, h] / np.sqrt(d)
            dv[s:e, hk] += P.T @ do[s:e, h]
    return dq, dk, dv
