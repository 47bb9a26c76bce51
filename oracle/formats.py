"""E4M3 element codes and UE8M0 power-of-two scales, written out from their definitions.

Source: "FLAMIA: FLAsh MIcroscaling Attention ..." Section 2 ("Microscaling
floating-point formats": MX blocks of 32 elements with UE8M0 scales, E4M3
codes), Section 3.2 (largest E4M3 value 448; the floor exponent rule of the
OCP reference conversion; the round-up rule that never clamps), Appendix A.5
(round to nearest).

E4M3 here is the "FN" variant used by MXFP8: 1 sign bit, 4 exponent bits with
bias 7, 3 mantissa bits; exponent field 0 holds subnormals m * 2^-9; there is
no infinity; 0x7F and 0xFF are NaN; the largest finite magnitude is
1.75 * 2^8 = 448.

Pinned by: exhaustive decode/encode round trip of all 254 finite codes,
hand-worked rounding cases (ties to even, subnormals, saturation), and an
in-range cross-check against torch.float8_e4m3fn (tests/test_oracle_formats.py).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_MIN_SUBNORMAL = 2.0 ** -9
E4M3_MIN_NORMAL = 2.0 ** -6
E4M3_BIAS = 7
UE8M0_BIAS = 127
SCALE_EXP_MIN = -127
SCALE_EXP_MAX = 127


def e4m3_decode_table() -> np.ndarray:
    """Value of every byte 0..255 (NaN for 0x7F/0xFF; 0x80 is -0.0)."""
    vals = np.empty(256, dtype=np.float64)
    for c in range(256):
        sign = -1.0 if (c & 0x80) else 1.0
        e = (c >> 3) & 0xF
        m = c & 0x7
        if e == 0xF and m == 0x7:
            vals[c] = np.nan
        elif e == 0:
            vals[c] = sign * m * E4M3_MIN_SUBNORMAL
        else:
            vals[c] = sign * (1.0 + m / 8.0) * 2.0 ** (e - E4M3_BIAS)
    return vals


_DECODE = e4m3_decode_table()


def e4m3_value(codes) -> np.ndarray:
    """Decode E4M3 bytes to float64."""
    return _DECODE[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(v) -> np.ndarray:
    """Round real values (given exactly as float64) to E4M3 bytes.

    Round to nearest, ties to the even code; magnitudes above 448 saturate to
    448 (finite saturation, no NaN); the sign is kept, so -0 and negative
    values that round to zero give 0x80.  Inputs must be finite.
    """
    v = np.asarray(v, dtype=np.float64)
    if not np.all(np.isfinite(v)):
        raise ValueError("E4M3 encode of a non-finite value")
    neg = np.signbit(v)
    a = np.abs(v)
    frac, ex = np.frexp(a)                     # a = frac * 2^ex, frac in [0.5, 1)
    e = np.where(a > 0, ex - 1, -1000)         # floor(log2 a)
    # spacing of representable values around a: 2^(e-3) in the normal range, 2^-9 below it
    q_exp = np.where(e >= -6, e - 3, -9)
    n = np.rint(np.ldexp(a, -q_exp))           # exact scaling, rint rounds half to even
    mag = np.minimum(np.ldexp(n, q_exp), E4M3_MAX)
    # magnitude -> code
    frac2, ex2 = np.frexp(mag)
    e2 = ex2 - 1
    normal = mag >= E4M3_MIN_NORMAL
    mant_n = np.where(normal, np.ldexp(mag, -e2) * 8.0 - 8.0, 0.0)
    code_n = ((e2 + E4M3_BIAS) << 3) + mant_n.astype(np.int64)
    code_s = np.ldexp(mag, 9).astype(np.int64)
    code = np.where(normal, code_n, code_s)
    code = np.where(neg, code | 0x80, code)
    return code.astype(np.uint8)


def quantize_value(v) -> np.ndarray:
    """E4M3 round trip: the value the code of ``v`` represents."""
    return e4m3_value(e4m3_encode(v))


def roundup_exponent(amax) -> np.ndarray:
    """Shared exponent of a block with maximum magnitude ``amax`` (Section 3.2).

    The scale's exponent is rounded up so the scaled maximum never exceeds 448:
    E is the smallest integer with amax <= 448 * 2^E.  Writing amax = m * 2^p
    with m in [1, 2): E = p - 8 if m <= 1.75, else p - 7.  E is clamped to the
    UE8M0 range [-127, 127]; an all-zero block gets E = -127.
    """
    a = np.asarray(amax, dtype=np.float64)
    frac, ex = np.frexp(a)
    p = ex - 1
    m = 2.0 * frac
    E = p - 8 + (m > 1.75).astype(np.int64)
    E = np.where(a > 0, E, SCALE_EXP_MIN)
    return np.clip(E, SCALE_EXP_MIN, SCALE_EXP_MAX).astype(np.int64)


def floor_exponent(amax) -> np.ndarray:
    """The OCP reference rule floor(log2 amax) - emax (emax = 8 for E4M3), Section 3.2.

    Kept only as the leaking negative control: the scaled maximum can reach
    [448, 512) and is then clamped to 448.
    """
    a = np.asarray(amax, dtype=np.float64)
    frac, ex = np.frexp(a)
    E = (ex - 1) - 8
    E = np.where(a > 0, E, SCALE_EXP_MIN)
    return np.clip(E, SCALE_EXP_MIN, SCALE_EXP_MAX).astype(np.int64)


def scale_byte(E) -> np.ndarray:
    """UE8M0 byte of the power-of-two scale 2^E."""
    return (np.asarray(E, dtype=np.int64) + UE8M0_BIAS).astype(np.uint8)


def bf16_round(x) -> np.ndarray:
    """Round float64 to the nearest bfloat16 value (ties to even), returned as float64.

    bfloat16 keeps 8 significant bits; its smallest normal is 2^-126 and the
    subnormal spacing below it is 2^-133.  Overflow is not handled (callers
    stay far inside the range).
    """
    x = np.asarray(x, dtype=np.float64)
    finite = np.isfinite(x)
    a = np.abs(np.where(finite, x, 0.0))
    frac, ex = np.frexp(a)
    e = np.maximum(ex - 1, -126)
    q_exp = e - 7
    mag = np.ldexp(np.rint(np.ldexp(a, -q_exp)), q_exp)
    out = np.where(np.signbit(x), -mag, mag)
    return np.where(finite, out, x)
