"""Pins for oracle.exact: textbook softmax, a library attention routine, finite differences, identities."""
import math

import numpy as np
import pytest
import torch

from oracle import exact as X


def _inputs(T, Hq, Hkv, d, seed=0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, Hq, d)); k = rng.standard_normal((T, Hkv, d))
    v = rng.standard_normal((T, Hkv, d)); do = rng.standard_normal((T, Hq, d))
    return q, k, v, do


def test_forward_matches_textbook_loops():
    cu = [0, 5, 12]
    q, k, v, _ = _inputs(12, 2, 1, 3, seed=1)
    O, lse = X.forward(q, k, v, cu)
    for (s, e) in [(0, 5), (5, 12)]:
        for h in range(2):
            for i in range(s, e):
                w = [math.exp(sum(q[i, h, c] * k[j, 0, c] for c in range(3)) / math.sqrt(3)) for j in range(s, i + 1)]
                Z = sum(w)
                for c in range(3):
                    o = sum(w[j - s] * v[j, 0, c] for j in range(s, i + 1)) / Z
                    assert abs(O[i, h, c] - o) < 1e-12
                assert abs(lse[h, i] - math.log(Z)) < 1e-12


@pytest.mark.parametrize("causal", [True, False])
def test_forward_matches_torch_sdpa_block_diagonal(causal):
    cu = [0, 30, 31, 64, 100]
    T, Hq, Hkv, d = 110, 4, 2, 16
    q, k, v, _ = _inputs(T, Hq, Hkv, d, seed=2)
    O, lse = X.forward(q, k, v, cu, causal=causal)
    mask = torch.zeros(T, T, dtype=torch.bool)
    for s, e in zip(cu[:-1], cu[1:]):
        blk = torch.ones(e - s, e - s, dtype=torch.bool)
        mask[s:e, s:e] = torch.tril(blk) if causal else blk
    tq = torch.from_numpy(q).permute(1, 0, 2)
    tk = torch.from_numpy(np.repeat(k, Hq // Hkv, axis=1)).permute(1, 0, 2)
    tv = torch.from_numpy(np.repeat(v, Hq // Hkv, axis=1)).permute(1, 0, 2)
    inside = slice(0, 100)
    ref = torch.nn.functional.scaled_dot_product_attention(tq[:, inside], tk[:, inside], tv[:, inside],
                                                           attn_mask=mask[inside, inside])
    assert np.allclose(O[inside].transpose(1, 0, 2), ref.numpy(), atol=1e-12, rtol=1e-12)
    assert np.all(O[100:] == 0) and np.all(np.isinf(lse[:, 100:]))


def test_gradients_match_finite_differences():
    cu = [0, 4, 9]
    T, Hq, Hkv, d = 9, 4, 2, 3
    q, k, v, do = _inputs(T, Hq, Hkv, d, seed=3)
    dq, dk, dv = X.backward(q, k, v, do, cu)

    def f(q_, k_, v_):
        return float((X.forward(q_, k_, v_, cu)[0] * do).sum())

    eps = 1e-6
    for name, arr, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            a1 = arr.copy(); a1[idx] += eps
            a2 = arr.copy(); a2[idx] -= eps
            args1 = {"q": q, "k": k, "v": v}; args1[name] = a1
            args2 = {"q": q, "k": k, "v": v}; args2[name] = a2
            num[idx] = (f(args1["q"], args1["k"], args1["v"]) - f(args2["q"], args2["k"], args2["v"])) / (2 * eps)
        rel = np.linalg.norm(num - grad) / np.linalg.norm(grad)
        assert rel < 1e-7, (name, rel)


def test_softmax_gradient_identities():
    # D_i = sum_j P_ij dP_ij = dO_i . O_i, and each row of dS sums to zero (Section 3.3)
    rng = np.random.default_rng(4)
    L, d = 20, 8
    q, k, v, do = (rng.standard_normal((L, d)) for _ in range(4))
    S = q @ k.T / math.sqrt(d)
    S = np.where(np.tril(np.ones((L, L), bool)), S, -np.inf)
    P = np.exp(S - S.max(1, keepdims=True)); P /= P.sum(1, keepdims=True)
    O = P @ v
    dP = do @ v.T
    D = (do * O).sum(1)
    assert np.allclose(D, (P * dP).sum(1), atol=1e-12)
    dS = P * (dP - D[:, None])
    assert np.allclose(dS.sum(1), 0.0, atol=1e-12)
