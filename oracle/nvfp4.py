"""NVFP4 operands of the mixed NVFP4/FP8 path: E2M1 element codes with one
UE4M3 scale per 16 consecutive head-dimension elements of each token.

Test infrastructure: imported only by tests, the smoke check and the CPU legs
of the benchmark.

Source: "FLAMIA: FLAsh MIcroscaling Attention ..." Section 3.4 (the mixed path
quantizes Q and K with one NVFP4 scale per 16 head-dimension elements of each
token; the same codes serve the forward scores and their recomputation in the
backward, the other products keep E4M3 operands), Section 3.2 (per-token NVFP4
scales cannot leak; scales are rounded so that no element is clamped) and
Appendix A.1 (the UE4M3 scale range).

E2M1: 1 sign bit, 2 exponent bits with bias 1, 1 mantissa bit; the
magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4 and 6; there is no infinity or NaN.
UE4M3: E4M3 without its sign bit (bytes 0x00 .. 0x7E), an unsigned block scale.

Readings where the pages leave it open:
  * no tensor-wide second-level scale (a whole-tensor statistic is the
    extreme leak of Section 3.2): a group's scale is its own UE4M3 value;
  * the scale is rounded up: the smallest UE4M3 value s with 6 s >= amax
    (6 s is exact), so |x| / s <= 6 and no element saturates; an all-zero
    group gets scale 0 and codes 0; amax > 6 * 448 saturates the scale at 448
    (its elements then saturate at 6);
  * an element's code is E2M1 round-to-nearest (ties to the even code) of the
    quotient x / s rounded once to fp32, as a kernel computes it; the sign is
    kept, so a negative value that rounds to zero gives the code 0x8.

Pinned by tests/test_oracle_nvfp4.py: the 16 codes round-trip, hand-worked
ties and saturation, a brute-force nearest-value search, the brute-force
scale search over all 127 UE4M3 values, the element error bound, and the
independence of tokens.
"""
from __future__ import annotations

import numpy as np

from .formats import e4m3_value

E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
E2M1_MAX = 6.0
GROUP = 16
UE4M3_VALUES = e4m3_value(np.arange(0x7F))        # 0 and the 126 positive finite E4M3 values, ascending


def e2m1_value(codes) -> np.ndarray:
    """Decode 4-bit E2M1 codes (one per byte, low nibble) to float64."""
    c = np.asarray(codes, dtype=np.uint8)
    mag = E2M1_MAGNITUDES[c & 0x7]
    return np.where(c & 0x8, -mag, mag)


def e2m1_encode(v) -> np.ndarray:
    """Round finite values to E2M1 codes: nearest magnitude, ties to the even
    code, saturating at 6, sign kept."""
    v = np.asarray(v, dtype=np.float64)
    if not np.all(np.isfinite(v)):
        raise ValueError("E2M1 encode of a non-finite value")
    a = np.minimum(np.abs(v), E2M1_MAX)
    hi = np.clip(np.searchsorted(E2M1_MAGNITUDES, a, side="left"), 1, 7)
    lo = hi - 1
    dlo = a - E2M1_MAGNITUDES[lo]
    dhi = E2M1_MAGNITUDES[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    mag_code = np.where(pick_hi, hi, lo)
    return (mag_code | np.where(np.signbit(v), 0x8, 0)).astype(np.uint8)


def ue4m3_roundup(amax):
    """Scale byte and value of a group with maximum magnitude ``amax``: the
    smallest UE4M3 value s with 6 s >= amax (0 for amax = 0, 448 above 6 * 448)."""
    a = np.asarray(amax, dtype=np.float64)
    idx = np.searchsorted(6.0 * UE4M3_VALUES, a, side="left")
    idx = np.minimum(idx, len(UE4M3_VALUES) - 1)
    return idx.astype(np.uint8), UE4M3_VALUES[idx]


def quantize_nvfp4(x, cu_seqlens):
    """NVFP4 codes of x [T, H, d] per (token, head, 16-element group).

    Returns (codes uint8 [T, H, d] one E2M1 code per byte, scale bytes uint8
    [T, H, d / 16], dequantized values float64 [T, H, d]).  Tokens outside every
    document keep codes 0 and scale 0.
    """
    x = np.asarray(x, dtype=np.float64)
    T, H, d = x.shape
    assert d % GROUP == 0
    codes = np.zeros((T, H, d), np.uint8)
    sbytes = np.zeros((T, H, d // GROUP), np.uint8)
    vals = np.zeros((T, H, d))
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    for r in range(len(cu) - 1):
        s, e = int(cu[r]), int(cu[r + 1])
        if e <= s:
            continue
        g = x[s:e].reshape(e - s, H, d // GROUP, GROUP)
        sb, sv = ue4m3_roundup(np.abs(g).max(axis=3))
        with np.errstate(divide="ignore", invalid="ignore"):
            quot = np.where(sv[..., None] > 0,
                            (g.astype(np.float32) / sv[..., None].astype(np.float32)).astype(np.float64), 0.0)
        c = e2m1_encode(quot)
        codes[s:e] = c.reshape(e - s, H, d)
        sbytes[s:e] = sb
        vals[s:e] = (e2m1_value(c) * sv[..., None]).reshape(e - s, H, d)
    return codes, sbytes, vals
