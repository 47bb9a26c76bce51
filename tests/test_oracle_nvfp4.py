"""Pins for oracle.nvfp4 and the mixed NVFP4/FP8 score path of oracle.simulated
(FLAMIA Sections 3.4 and 3.5.2, Appendix A.1, Table 4)."""
import json
import os

import numpy as np
import pytest

from oracle import exact as X
from oracle import formats as F
from oracle import nvfp4 as N
from oracle import simulated as S

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "paper_facts.json")))


def test_e2m1_codes_round_trip():
    for c in range(16):
        assert N.e2m1_encode(N.e2m1_value(c))[()] == c
    assert list(N.e2m1_value(np.arange(8))) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_hand_cases():
    # ties go to the even code; above 6 saturates; the sign is kept
    cases = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6, 5.01: 7, 7.0: 7, 1e9: 7,
             0.2: 0, 0.3: 1, -0.1: 8, -5.5: 15}
    for v, c in cases.items():
        assert N.e2m1_encode(v)[()] == c, v


def test_e2m1_nearest_by_brute_force():
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.uniform(-7, 7, 5000), np.arange(-14, 15) * 0.25])
    got = N.e2m1_encode(v)
    for x, c in zip(v, got):
        a = min(abs(x), 6.0)
        d = [abs(a - m) for m in (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)]
        best = [i for i in range(8) if d[i] == min(d)]
        want = [i for i in best if i % 2 == 0][0] if len(best) > 1 else best[0]
        assert c & 7 == want and bool(c & 8) == bool(np.signbit(x)), x


def test_ue4m3_scale_is_smallest_admissible_by_search():
    rng = np.random.default_rng(1)
    amax = np.concatenate([np.exp2(rng.uniform(-14, 12, 3000)), 6.0 * F.e4m3_value(np.arange(1, 127)), [0.0]])
    positive = sorted(v for v in F.e4m3_value(np.arange(0x80)) if np.isfinite(v) and v > 0)
    sb, sv = N.ue4m3_roundup(amax)
    for a, b, s in zip(amax, sb, sv):
        if a == 0:
            assert b == 0 and s == 0
            continue
        fit = [v for v in positive if 6.0 * v >= a]
        want = fit[0] if fit else 448.0
        assert s == want and F.e4m3_value(b) == s, a


def test_nvfp4_error_bound_and_groups():
    rng = np.random.default_rng(2)
    x = F.bf16_round(rng.standard_normal((40, 3, 64)) * np.exp2(rng.integers(-8, 8, (40, 3, 4)).repeat(16, axis=2)))
    codes, sb, vals = N.quantize_nvfp4(x, [0, 40])
    s = F.e4m3_value(sb).repeat(16, axis=2)
    # |x| / s <= 6 (no element clamped) and the error is at most half the
    # widest E2M1 gap (between 4 and 6) in units of the scale, plus one fp32
    # rounding of the quotient
    assert np.all(np.abs(x) <= 6.0 * s)
    assert np.all(np.abs(vals - x) <= s * (1.0 + 1e-6))
    # each 16-element group uses its own scale: rescaling one group by 2^k
    # rescales only its own values
    x2 = x.copy(); x2[5, 1, 16:32] *= 8.0
    v2 = N.quantize_nvfp4(x2, [0, 40])[2]
    changed = np.argwhere(v2 != vals)
    assert changed.size and np.all(changed[:, 0] == 5) and np.all(changed[:, 1] == 1)
    assert np.all((changed[:, 2] >= 16) & (changed[:, 2] < 32))


def test_nvfp4_tokens_and_documents_are_independent():
    rng = np.random.default_rng(3)
    x = F.bf16_round(rng.standard_normal((50, 2, 32)))
    c0, s0, _ = N.quantize_nvfp4(x, [0, 20, 50])
    x2 = x.copy(); x2[30] *= 1e3
    c1, s1, _ = N.quantize_nvfp4(x2, [0, 20, 50])
    keep = np.arange(50) != 30
    assert np.array_equal(c0[keep], c1[keep]) and np.array_equal(s0[keep], s1[keep])


@pytest.mark.parametrize("causal", [True, False])
def test_nvfp4_path_without_quantizers_is_exact_attention(causal):
    rng = np.random.default_rng(4)
    f = lambda shp: F.bf16_round(rng.standard_normal(shp))
    q, k, v, do = f((300, 2, 32)), f((300, 1, 32)), f((300, 1, 32)), f((300, 2, 32))
    cu = [0, 170, 300]
    Ox, lx = X.forward(q, k, v, cu, causal=causal)
    r = S.forward(q, k, v, cu, causal=causal, scores="nvfp4", quantize=False, p_quant=False)
    assert np.allclose(r["O"], Ox, rtol=1e-12, atol=1e-12)


def test_log_domain_p_hat_uses_the_group_maximum():
    """Every (row, 32-key group) scale is the round-up exponent of the group's
    largest probability, so the largest P-hat input of a call lies in
    (224, 448]: above half the largest code, never above it."""
    rng = np.random.default_rng(5)
    f = lambda shp: F.bf16_round(rng.standard_normal(shp))
    q, k, v = f((260, 2, 64)), f((260, 1, 64)), f((260, 1, 64))
    r = S.forward(q, k, v, [0, 260], scores="nvfp4")
    assert 224.0 < r["pmax"] <= 448.0
    # and so does every (row, group) that sees a key, however far below the
    # row maximum its probabilities are
    assert 224.0 < r["p_group_max_min"] <= 448.0
    r8 = S.forward(q, k, v, [0, 260])                # the fixed 2^c multiplier stays below 2^(c + tau)
    assert r8["pmax"] <= 256.0 and r8["p_group_max_min"] < 224.0


def test_gradient_products_keep_e4m3_operands():
    """dQ and dK contract the E4M3 token-block K and Q, not the NVFP4 copies:
    with one outlier channel per 16-element group, NVFP4 flushes the other
    channels of Q and K, yet the gradients on those channels stay as close to
    exact attention as the score error allows."""
    rng = np.random.default_rng(6)
    T, d = 256, 64

    def outliers(x):
        x = x.copy(); x[:, :, ::16] *= 12.0
        return F.bf16_round(x)
    q = outliers(rng.standard_normal((T, 2, d)) * 0.3)
    k = outliers(rng.standard_normal((T, 1, d)) * 0.3)
    v = F.bf16_round(rng.standard_normal((T, 1, d)))
    do = F.bf16_round(rng.standard_normal((T, 2, d)))
    gx = X.backward(q, k, v, do, [0, T])
    fo = S.forward(q, k, v, [0, T], scores="nvfp4")
    b = S.backward(q, k, v, fo["O_bf16"], fo["lse"], do, [0, T], scores="nvfp4")
    small = np.ones(d, bool); small[::16] = False
    rel = lambda a, c: np.linalg.norm(a - c) / np.linalg.norm(c)
    assert rel(b["dk"][:, :, small], gx[1][:, :, small]) < 0.25
    assert rel(b["dq"][:, :, small], gx[0][:, :, small]) < 0.25


@pytest.mark.parametrize("causal", [True, False])
def test_cosines_match_table4(causal):
    """Gaussian bf16 inputs at d = 128 (2 heads, 2 x 512 tokens): the mixed
    NVFP4/FP8 path's O and dQ cosines to exact attention fall within 0.002 of
    the paper's Table 4, and the MXFP8 path's O cosine within its 8-bit band."""
    t4 = GOLDEN["table4_cosines"]
    rng = np.random.default_rng(0)
    f = lambda shp: F.bf16_round(rng.standard_normal(shp))
    q, k, v, do = f((1024, 2, 128)), f((1024, 2, 128)), f((1024, 2, 128)), f((1024, 2, 128))
    cu = [0, 512, 1024]
    cos = lambda a, b: float((a * b).sum() / np.linalg.norm(a) / np.linalg.norm(b))
    Ox, _ = X.forward(q, k, v, cu, causal=causal)
    gx = X.backward(q, k, v, do, cu, causal=causal)
    fo = S.forward(q, k, v, cu, causal=causal, scores="nvfp4")
    b = S.backward(q, k, v, fo["O_bf16"], fo["lse"], do, cu, causal=causal, scores="nvfp4")
    want = t4["nvfp4_fp8_causal" if causal else "nvfp4_fp8_noncausal"]
    assert abs(cos(fo["O"], Ox) - want[0]) <= 2e-3
    assert abs(cos(b["dq"], gx[0]) - want[1]) <= 2e-3
    f8 = S.forward(q, k, v, cu, causal=causal)
    lo, hi = t4["eight_bit_o_range"]
    assert lo - 1e-3 <= cos(f8["O"], Ox) <= hi + 1e-3
