"""Hadamard rotation of Q and K along the head dimension.

Test infrastructure: imported only by tests, the smoke check and the CPU legs
of the benchmark.

Source: "FLAMIA: FLAsh MIcroscaling Attention ..." Section 3.4 and Appendix
A.2: a Hadamard transform mixes the head channels of both Q and K before
quantization; the shared orthogonal transform leaves Q K^T unchanged in exact
arithmetic and spreads channel outliers over all channels of a block.

Readings where the pages leave it open:
  * the transform is the Sylvester Hadamard matrix H_n (entries +-1, n = d),
    not normalized; H_n H_n^T = n I, so scores computed from rotated operands
    carry a factor n, taken out exactly (a power of two) with the softmax
    scale, and the gradients of the rotated operands map back with H_n / n;
  * the rotation is computed in fp32, by radix-2 butterflies with strides
    1, 2, 4, ..., n/2 in that order, the lower element of each pair first
    ((a, b) -> (a + b, a - b)); the quantizer codes the fp32 results.  The
    order fixes the fp32 roundings, so codes are reproducible bit for bit.

Pinned by tests/test_oracle_hadamard.py: the butterflies against an explicit
matrix product with scipy.linalg.hadamard on small integers (exact), the
rotation's orthogonality, and the reduction of the rotated simulated
attention to exact attention when every quantizer is off.
"""
from __future__ import annotations

import numpy as np


def sylvester(n: int) -> np.ndarray:
    """H_n by the Sylvester construction (n a power of two), float64."""
    assert n >= 1 and n & (n - 1) == 0
    h = np.ones((1, 1))
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def fwht_fp32(x) -> np.ndarray:
    """x @ H_n along the last axis, in float32 by radix-2 butterflies (see module doc)."""
    y = np.array(x, dtype=np.float32, copy=True)
    n = y.shape[-1]
    assert n & (n - 1) == 0
    lead = y.shape[:-1]
    h = 1
    while h < n:
        v = y.reshape(lead + (n // (2 * h), 2, h))
        a = v[..., 0, :].copy()
        b = v[..., 1, :].copy()
        v[..., 0, :] = a + b
        v[..., 1, :] = a - b
        y = v.reshape(lead + (n,))
        h *= 2
    return y


def rotate(x) -> np.ndarray:
    """Rotated operand [T, H, d] as float64 values of the fp32 butterflies."""
    return fwht_fp32(np.asarray(x, np.float32)).astype(np.float64)


def unrotate(g) -> np.ndarray:
    """Gradient of a rotated operand mapped back: g H_n / n, exact in fp64."""
    g = np.asarray(g, np.float64)
    n = g.shape[-1]
    return (g @ sylvester(n)) / n
