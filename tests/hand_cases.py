"""Hand-worked inputs whose outputs are derived on paper, for pins of the oracle
and of the CUDA path.  Only tests import this module; it holds input data and
the hand-derived expected values, none of the method's arithmetic.

Two-token document (tokens 0 and 1 of a 128-token row; tokens 2..127 belong to
no document), one head, d = 64 (the numbers below) or d = 128.  Every input value is exactly representable
after its document-local 32-token block quantization (FLAMIA Section 3.1,
round-up exponent of Section 3.2):
  * q0 = q1 = 1 in every channel (block max 1: exponent -8, codes 256);
  * k0: six channels -2 and 58 channels -1, so q.k0 = -70; k1 = 0 (block max
    2: exponent -7, codes -256 and -128);
  * v0 = 1, v1 = 0 (exponent -8);
  * dO0 = 0, dO1 = 1 (exponent -8).
With the softmax scale log2(e)/sqrt(64), row 1 sees the scores (in log2 units)
S = -70 log2(e) / 8 = -12.62358... for key 0 and 0 for key 1; row 0 sees only
key 0.  At d = 128, k0 has 99 channels -1 and 29 zeros (exponent -8), q.k0 =
-99 and S = -99 log2(e) / sqrt(128) = -12.62423..., which lands in the same
rounding windows (2^S = 1.2975 * 2^-13), so every statement below holds with
that S.

Forward, row 1 (one key tile; m = 0): p~ = (2^S, 1), and 2^S = 1.29812 * 2^-13.
  * P-hat with c = 4: E4M3(16 * 2^S) = E4M3(1.298 * 2^-9) lies on the
    subnormal grid of step 2^-9 and rounds to 2^-9, so P-hat = 2^-13; the
    other key gives E4M3(16) / 16 = 1.
  * The row sum accumulates the unquantized p~ (Section 3.3: quantized
    probabilities need not sum to one): l = 1 + 2^S.
  * O1 = (2^-13 v0 + 1 v1) / l = 2^-13 / (1 + 2^S) in every channel, and
    LSE1 = ln(1 + 2^S).  Had l summed the P-hat values instead, LSE1 would be
    ln(1 + 2^-13), 3.6e-5 lower.
Row 0: O0 = v0 = 1 and LSE0 = S ln 2 = -8.75.

Backward: P10 = 2^(S - log2(1 + 2^S)) = 2^S / (1 + 2^S).  The dV operand is
E4M3(2^8 P) 2^-8 (Appendix B.1): 2^8 P10 = 1.2979 * 2^-5 lies between the
E4M3 neighbours 1.25 * 2^-5 and 1.375 * 2^-5 and rounds to the first, so
dV0 = P'10 dO1 + P'00 dO0 = 1.25 * 2^-13 in every channel (exact in bf16).
With a multiplier of 2^4 instead, 2^4 P10 = 1.298 * 2^-9 would round to 2^-9
on the subnormal grid (dV0 = 2^-13); with none, P10 would round to 0.
"""
from __future__ import annotations

import math
import types

import numpy as np

T = 128
CU_SEQLENS = np.array([0, 2], np.int32)
DOT = {64: -70.0, 128: -99.0}


def values(d: int = 64):
    """The hand-derived outputs for head dimension d."""
    s = DOT[d] * math.log2(math.e) / math.sqrt(d)
    return types.SimpleNamespace(
        S_LOG2=s,
        LSE0=s * math.log(2.0),                           # -8.75 at d = 64
        LSE1=math.log1p(2.0 ** s),
        LSE1_IF_L_SUMMED_PHAT=math.log1p(2.0 ** -13),
        O1=2.0 ** -13 / (1.0 + 2.0 ** s),
        DV0=1.25 * 2.0 ** -13,
        DV0_IF_MULTIPLIER={8: 1.25 * 2.0 ** -13, 4: 2.0 ** -13, 0: 0.0},
    )


def arrays(d: int = 64):
    """q, k, v, dO as float64 [T, 1, d] arrays."""
    q = np.zeros((T, 1, d)); k = np.zeros((T, 1, d))
    v = np.zeros((T, 1, d)); do = np.zeros((T, 1, d))
    q[0:2, 0, :] = 1.0
    if d == 64:
        k[0, 0, :] = -1.0
        k[0, 0, :6] = -2.0
    else:
        k[0, 0, :99] = -1.0
    v[0, 0, :] = 1.0
    do[1, 0, :] = 1.0
    assert q[1, 0] @ k[0, 0] == DOT[d]
    return q, k, v, do


def workload(d: int = 64):
    """The same inputs as a workload record (bf16 tensors) for the GPU helpers."""
    import torch
    q, k, v, do = arrays(d)
    tens = {n: torch.from_numpy(x).to(torch.bfloat16) for n, x in zip(("q", "k", "v", "do"), (q, k, v, do))}
    return types.SimpleNamespace(tensors=tens, cu_seqlens=CU_SEQLENS, n_docs=1, T=T, Hq=1, Hkv=1, d=d)
