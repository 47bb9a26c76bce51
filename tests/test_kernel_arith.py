"""Identities the CUDA kernels rely on, checked in float32 on the host.

The kernels scale the score accumulators by x * 2^e (x = log2(e)/sqrt(d) or 1,
e the sum of two UE8M0 exponents, so e in [-254, 254]) without a branch:
x * 2^(e>>1) * 2^(e - (e>>1)), each factor built from its exponent bits (a
factor 2^-127 has a zero exponent field and reads as 0).  That must equal a
single correctly rounded x * 2^e for every e of the range.
"""
import numpy as np
import pytest


def pow2f(k: int) -> np.float32:
    # the kernels' bit construction: exponent field k + 127, zero mantissa
    return np.array([(k + 127) << 23], dtype=np.uint32).view(np.float32)[0]


def split_scale(x: np.float32, e: int) -> np.float32:
    e1 = e >> 1
    with np.errstate(over="ignore", under="ignore"):
        return np.float32(np.float32(x * pow2f(e1)) * pow2f(e - e1))


@pytest.mark.parametrize("x", [0.18033688011112042, 0.12751743082459868, 1.0])
def test_split_power_of_two_scaling_is_ldexp(x):
    xf = np.float32(x)
    for e in range(-254, 255):
        with np.errstate(over="ignore", under="ignore"):
            want = np.ldexp(xf, e).astype(np.float32)
        got = split_scale(xf, e)
        assert got == want or (np.isinf(got) and np.isinf(want)), (x, e, got, want)


def test_pow2f_bits():
    assert pow2f(0) == 1.0 and pow2f(127) == 2.0 ** 127 and pow2f(-126) == 2.0 ** -126
    assert pow2f(-127) == 0.0
