"""Pins for oracle.hadamard and the rotated simulated attention (FLAMIA Section 3.4,
Appendix A.2): the fp32 butterflies against an explicit matrix product, the
Sylvester matrix against a library construction, and the reduction of the
rotated path to exact attention when no quantizer is applied."""
import numpy as np
import pytest

from oracle import exact as X
from oracle import formats as F
from oracle import hadamard as HD
from oracle import simulated as S


@pytest.mark.parametrize("n", [2, 8, 64, 128])
def test_sylvester_matches_library_and_is_orthogonal_up_to_n(n):
    linalg = pytest.importorskip("scipy.linalg")
    H = HD.sylvester(n)
    assert np.array_equal(H, linalg.hadamard(n).astype(np.float64))
    assert np.array_equal(H @ H.T, n * np.eye(n))
    assert np.array_equal(H, H.T)


@pytest.mark.parametrize("n", [8, 128])
def test_butterflies_equal_matrix_product_on_small_integers(n):
    # integers below 2^10: every partial sum is exact in fp32, so the butterflies
    # must reproduce x @ H exactly
    rng = np.random.default_rng(0)
    x = rng.integers(-1000, 1000, size=(5, 3, n)).astype(np.float64)
    got = HD.fwht_fp32(x).astype(np.float64)
    assert np.array_equal(got, x @ HD.sylvester(n))
    assert np.array_equal(HD.unrotate(got), x)


def test_butterfly_order_fixes_the_fp32_roundings():
    # values whose sums round in fp32: the stride order 1, 2, 4, ... is part of the
    # definition, and another order gives other bits somewhere
    rng = np.random.default_rng(1)
    x = F.bf16_round(rng.standard_normal((64, 128)) * np.exp2(rng.integers(-12, 12, (64, 128))))
    y = HD.fwht_fp32(x)
    exact = x @ HD.sylvester(128)
    # fp32 rounding of sums of 128 terms: relative to each row's size
    assert np.max(np.linalg.norm(y - exact, axis=1) / np.linalg.norm(exact, axis=1)) < 1e-6
    # reversed stride order
    z = np.array(x, np.float32)
    h = 64
    while h >= 1:
        v = z.reshape(64, 128 // (2 * h), 2, h)
        a, b = v[:, :, 0, :].copy(), v[:, :, 1, :].copy()
        v[:, :, 0, :], v[:, :, 1, :] = a + b, a - b
        z = v.reshape(64, 128)
        h //= 2
    assert not np.array_equal(y, z)


CU = [0, 200, 333, 600]


def _inputs(seed, d=128):
    rng = np.random.default_rng(seed)
    f = lambda shp: F.bf16_round(rng.standard_normal(shp))
    return f((600, 2, d)), f((600, 1, d)), f((600, 1, d)), f((600, 2, d))


def test_rotated_forward_without_quantizers_is_exact_attention():
    q, k, v, _ = _inputs(2)
    Ox, lx = X.forward(q, k, v, CU)
    r = S.forward(q, k, v, CU, quantize=False, p_quant=False, exact_max=True, hadamard=True)
    assert np.allclose(r["O"], Ox, rtol=1e-5, atol=1e-6)
    assert np.allclose(r["lse"][:, :600], lx[:, :600], rtol=1e-6, atol=1e-6)


def test_rotated_backward_without_quantizers_is_exact_gradient():
    q, k, v, do = _inputs(3)
    Ox, lx = X.forward(q, k, v, CU)
    gx = X.backward(q, k, v, do, CU)
    r = S.backward(q, k, v, Ox, lx, do, CU, quantize=False, p_quant=False, ds_quant=False, hadamard=True)
    for a, b in zip((r["dq"], r["dk"], r["dv"]), gx):
        assert np.allclose(a, b, rtol=1e-4, atol=1e-5)


def test_rotation_adds_no_cross_document_channel():
    # the rotation mixes channels of one token, never tokens: scaling another
    # document changes no bit of this document's rotated codes or outputs
    cu = [0, 150, 420, 600]
    q, k, v, do = _inputs(5)
    f0 = S.forward(q, k, v, cu, hadamard=True)
    b0 = S.backward(q, k, v, f0["O_bf16"], f0["lse"], do, cu, hadamard=True)
    q2, k2, v2, do2 = (x.copy() for x in (q, k, v, do))
    for x in (q2, k2, v2, do2):
        x[150:420] *= 1e4
    f1 = S.forward(q2, k2, v2, cu, hadamard=True)
    b1 = S.backward(q2, k2, v2, f1["O_bf16"], f1["lse"], do2, cu, hadamard=True)
    for sl in (slice(0, 150), slice(420, 600)):
        assert np.array_equal(f0["q"][1][sl], f1["q"][1][sl])
        assert np.array_equal(f0["O"][sl], f1["O"][sl])
        for key in ("dq", "dk", "dv"):
            assert np.array_equal(b0[key][sl], b1[key][sl])
