"""Hand-worked pins of two parts of the simulating oracle (oracle.simulated)
that Gaussian inputs and tolerances cannot tell apart from plausible mistakes:

  * the dV operand's probability multiplier 2^8 (FLAMIA Appendix B.1: the
    backward multiplies P by 2^8 before its E4M3 rounding and stores no scale);
  * the row sum over the unquantized p~ (FLAMIA Section 3.3: quantized
    probabilities need not sum to one, so l is not the sum of the P-hat values).

The inputs and the values they must give are derived by hand in
tests/hand_cases.py.  Each planted mistake (multiplier 2^4 or 2^0; l summed
over P-hat) moves an output far beyond the tolerance used here.
"""
import inspect
import json
import math
import pathlib

import numpy as np
import pytest

from oracle import simulated as OS
from tests import hand_cases as HC

FACTS = json.loads((pathlib.Path(__file__).parent / "golden" / "paper_facts.json").read_text())


def _run(d, p_bwd_exp=None):
    q, k, v, do = HC.arrays(d)
    f = OS.forward(q, k, v, HC.CU_SEQLENS)
    kw = {} if p_bwd_exp is None else {"p_bwd_exp": p_bwd_exp}
    b = OS.backward(q, k, v, f["O_bf16"], f["lse"], do, HC.CU_SEQLENS, **kw)
    return f, b


@pytest.mark.parametrize("d", [64, 128])
def test_forward_row_sum_is_over_unquantized_probabilities(d):
    hv = HC.values(d)
    f, _ = _run(d)
    O, lse = f["O"], f["lse"]
    assert np.allclose(O[0, 0], 1.0, rtol=0, atol=1e-15)
    assert abs(lse[0, 0] - hv.LSE0) < 1e-12
    assert np.allclose(O[1, 0], hv.O1, rtol=1e-12, atol=0)
    assert abs(lse[0, 1] - hv.LSE1) < 1e-14
    # the mistaken convention (l = sum of P-hat) is far outside that tolerance
    assert abs(hv.LSE1 - hv.LSE1_IF_L_SUMMED_PHAT) > 3e-5
    # rows outside the document
    assert np.all(O[2:] == 0) and np.all(np.isinf(lse[0, 2:]))


@pytest.mark.parametrize("d", [64, 128])
def test_dv_operand_multiplier_is_two_to_the_eight(d):
    facts_exp = FACTS["dv_probability_multiplier"]["exponent"]
    default = inspect.signature(OS.backward).parameters["p_bwd_exp"].default
    assert default == facts_exp == 8
    hv = HC.values(d)
    _, b = _run(d)
    assert np.allclose(b["dv"][0, 0], hv.DV0, rtol=1e-12, atol=0)
    assert np.all(b["dv_bf16"][0, 0] == hv.DV0)            # exact in bf16


@pytest.mark.parametrize("d", [64, 128])
def test_dv_pin_catches_other_multipliers(d):
    hv = HC.values(d)
    for e in (4, 0):
        _, b = _run(d, p_bwd_exp=e)
        assert np.allclose(b["dv"][0, 0], hv.DV0_IF_MULTIPLIER[e], rtol=1e-12, atol=0), e
        assert abs(b["dv"][0, 0, 0] - hv.DV0) > 0.15 * hv.DV0, e


@pytest.mark.parametrize("d", [64, 128])
def test_hand_values(d):
    # 2^S sits where the derivation says: 16 * 2^S rounds to 2^-9 on the
    # E4M3 subnormal grid, and 2^8 P10 rounds to 1.25 * 2^-5
    hv = HC.values(d)
    x = 2.0 ** hv.S_LOG2
    assert 1.29 * 2.0 ** -13 < x < 1.31 * 2.0 ** -13
    assert round(16 * x / 2.0 ** -9) == 1
    p10 = x / (1 + x)
    m = 2.0 ** 8 * p10 / 2.0 ** -5                     # significand on the 1/8 grid of [1, 2)
    assert abs(m - 1.25) < abs(m - 1.375) and m > 1.25
    assert math.isclose(hv.O1, 2.0 ** -13 / (1 + x))
    if d == 64:
        assert abs(hv.LSE0 + 8.75) < 1e-12
