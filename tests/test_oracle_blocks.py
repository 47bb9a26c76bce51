"""Pins for oracle.blocks: document-local 32-token blocks with round-up exponents."""
import numpy as np
import pytest

from oracle import blocks as B
from oracle import formats as F


def test_block_boundaries_hand_listed():
    got = [(b0, b1) for _, b0, b1 in B.doc_blocks([0, 96, 160, 256])]
    assert got == [(0, 32), (32, 64), (64, 96), (96, 128), (128, 160), (160, 192), (192, 224), (224, 256)]
    got = [(r, b0, b1) for r, b0, b1 in B.doc_blocks([0, 40, 40, 45, 110])]
    assert got == [(0, 0, 32), (0, 32, 40), (2, 40, 45), (3, 45, 77), (3, 77, 109), (3, 109, 110)]


def _rand(T, H, d, seed=0, scale=1.0):
    rng = np.random.default_rng(seed)
    return F.bf16_round(rng.standard_normal((T, H, d)) * scale)


def test_block_exponent_is_smallest_admissible():
    cu = [0, 50, 77, 200]
    x = _rand(200, 3, 16)
    codes, sb, E = B.quantize_token_blocks(x, cu)
    for r, b0, b1 in B.doc_blocks(cu):
        for h in range(3):
            amax = np.abs(x[b0:b1, h]).max()
            cand = [e for e in range(-127, 128) if amax <= 448.0 * 2.0 ** e]
            assert np.all(E[h, b0:b1] == min(cand))
            assert np.all(sb[h, b0:b1] == min(cand) + 127)
            vals = F.e4m3_value(codes[b0:b1, h])
            assert np.abs(vals).max() <= 448.0
            # exponent minimal => the block maximum lands in the top binade range (224, 448]
            assert np.abs(vals).max() > 224.0


def test_dequantized_error_bound():
    cu = [0, 128]
    x = _rand(128, 2, 32, seed=4)
    codes, _, E = B.quantize_token_blocks(x, cu)
    xh = B.dequantize(codes, E)
    # E4M3 normal relative error <= 2^-4; subnormal absolute error <= 2^-10 * 2^E
    bound = np.maximum(np.abs(x) * 2.0 ** -4, np.ldexp(2.0 ** -10, E.T[:, :, None]))
    assert np.all(np.abs(xh - x) <= bound * (1 + 1e-12))


@pytest.mark.parametrize("k", [-20, -3, 1, 7])
def test_power_of_two_shift_invariance(k):
    cu = [0, 70, 100]
    x = _rand(100, 2, 8, seed=5)
    c0, _, E0 = B.quantize_token_blocks(x, cu)
    c1, _, E1 = B.quantize_token_blocks(np.ldexp(x, k), cu)
    assert np.array_equal(c0, c1) and np.array_equal(E1, E0 + k)


def test_documents_are_independent():
    cu = [0, 37, 90, 160]
    x = _rand(160, 2, 8, seed=6)
    y = x.copy()
    y[37:90] *= 1e4                                  # perturb only document 1
    c0, s0, _ = B.quantize_token_blocks(x, cu)
    c1, s1, _ = B.quantize_token_blocks(y, cu)
    for sl in (slice(0, 37), slice(90, 160)):
        assert np.array_equal(c0[sl], c1[sl]) and np.array_equal(s0[:, sl], s1[:, sl])


def test_outside_documents_untouched():
    cu = [0, 20]
    x = _rand(40, 1, 8, seed=7)
    c, s, E = B.quantize_token_blocks(x, cu)
    assert np.all(c[20:] == 0) and np.all(E[:, 20:] == -127)
