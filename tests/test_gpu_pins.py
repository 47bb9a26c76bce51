"""GPU pins that need no tolerance argument.

* The hand-worked two-token case of tests/hand_cases.py run through the C ABI:
  the CUDA forward's LSE follows the row sum over unquantized probabilities
  (FLAMIA Section 3.3) and is far from the value a P-hat sum would give; the
  CUDA backward's dV operand carries the 2^8 multiplier (Appendix B.1), so
  dV0 is exactly 1.25 * 2^-13.
* flamia_quantize on its own (Section 3.1 token blocks, Section 3.2 round-up
  exponent, Section 3.6.1 document-local blocks on the packed layout): codes
  and scale bytes bit-exact against the oracle's block quantizer on a ragged
  packed row with tokens outside every document at both ends.
"""
import numpy as np
import pytest
import torch

import precision_causal_attention_gb300 as F
from oracle import blocks as OB
from tests import hand_cases as HC
from tests.gpu_common import run_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d", [64, 128])
def test_hand_case_row_sum_and_dv_multiplier(d):
    hv = HC.values(d)
    res = run_gpu(HC.workload(d))
    assert res["status"] == 0
    lse, out, dv = res["lse"], res["out"], res["dv"]
    # row 0 sees only key 0: O0 = v0 = 1, LSE0 = S ln 2
    assert np.all(out[0, 0] == 1.0)
    assert abs(lse[0, 0] - hv.LSE0) < 1e-5
    # row 1: LSE from l = 1 + 2^S (the P-hat sum would give 3.6e-5 less)
    assert abs(lse[0, 1] - hv.LSE1) < 5e-6, (lse[0, 1], hv.LSE1)
    assert abs(lse[0, 1] - hv.LSE1_IF_L_SUMMED_PHAT) > 2.5e-5
    # O1 = 2^-13 / (1 + 2^S) rounds to 2^-13 in bf16
    assert np.all(out[1, 0] == 2.0 ** -13)
    # dV0 = E4M3(2^8 P10) 2^-8 exactly; 2^4 would give 2^-13, no multiplier 0
    assert np.all(dv[0, 0] == hv.DV0), dv[0, 0, :4]
    # rows outside the document
    assert np.all(out[2:] == 0) and np.all(np.isinf(lse[0, 2:]))
    for key in ("dq", "dk", "dv"):
        assert np.all(res[key][2:] == 0), key


@pytest.mark.parametrize("d", [64, 128])
def test_flamia_quantize_standalone_bit_exact(d):
    dev = torch.device("cuda:0")
    T, H = 700, 3
    cu_np = np.array([5, 305, 322, 451, 451, 651], np.int32)    # tokens 0..4 and 651..699 outside
    g = torch.Generator().manual_seed(21 + d)
    x = torch.randn(T, H, d, generator=g)
    # per-token magnitudes over many binades, so blocks take many exponents
    x *= torch.pow(2.0, torch.randint(-20, 20, (T, 1, 1), generator=g).float())
    x = x.to(torch.bfloat16)
    cu = torch.from_numpy(cu_np).to(dev)
    xd = x.to(dev)
    for rep in range(2):
        codes = torch.full((T, H, d), 0xAB, dtype=torch.uint8, device=dev)
        scales = torch.full((H, T), 0xAB, dtype=torch.uint8, device=dev)
        F.flamia_quantize(xd, cu, codes, scales)
        assert F.flamia_last_launch_count() == 1
        torch.cuda.synchronize()
        assert F.flamia_get_status() == 0
        want_codes, want_scales, _ = OB.quantize_token_blocks(x.float().numpy().astype(np.float64), cu_np)
        assert np.array_equal(codes.cpu().numpy(), want_codes), rep
        assert np.array_equal(scales.cpu().numpy(), want_scales), rep
        # tokens outside every document: code 0, scale byte 0
        assert not codes[:5].any() and not codes[651:].any()
        assert not scales[:, :5].any() and not scales[:, 651:].any()
