"""GPU parity of the mixed NVFP4/FP8 path (flamia_opts.nvfp4) against the oracle.

FLAMIA Section 3.4: the forward's scores and their recomputation in the
backward multiply NVFP4 Q and K (E2M1 codes, one UE4M3 scale per 16
head-dimension elements of each token) with a block-scaled 4-bit MMA; every
other product keeps the E4M3 token-block operands.  Section 3.5.2: P-hat is
quantized in the log domain, one exponent per (query row, 32-key group).

Bar: the NVFP4 codes and scales of Q and K, and the E4M3 codes and scales of
Q, K, V and dO, bit-exact; O and LSE within 1e-2 and dQ, dK, dV within 3e-2
(relative Frobenius) of the simulating oracle with scores="nvfp4".  The
cosine to exact fp64 attention is reported next to the oracle's own.
"""
import numpy as np
import pytest

import workloads as W
from oracle import blocks as OB
from oracle import exact as OX
from oracle import nvfp4 as ON
from oracle import simulated as OS
from tests.gpu_common import run_gpu, np_inputs, rel_fro, cosine

pytestmark = pytest.mark.gpu

FWD_TOL = 1e-2
BWD_TOL = 3e-2

CASES = [
    ("ragged_d64_gqa", lambda: W.custom([300, 17, 129, 0, 256, 1, 40], Hq=4, Hkv=2, d=64, seed=31, T=800)),
    ("ragged_d128", lambda: W.custom([260, 128, 33, 400], Hq=2, Hkv=1, d=128, seed=32, T=840)),
]


def _unpack(packed):
    """[T, H, d/2] bytes -> [T, H, d] codes, element 2i from the low nibble."""
    return np.stack([packed & 0xF, packed >> 4], axis=-1).reshape(packed.shape[0], packed.shape[1], -1)


@pytest.mark.parametrize("name,make", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("causal", [True, False])
def test_nvfp4_path_parity(name, make, causal):
    w = make()
    res = run_gpu(w, causal=causal, nvfp4=True)
    assert res["status"] == 0
    x = np_inputs(w)
    # NVFP4 Q and K, bit-exact (tokens outside every document: codes 0, scales 0)
    for key in ("q", "k"):
        codes, sbytes, _ = ON.quantize_nvfp4(x[key], w.cu_seqlens)
        assert np.array_equal(_unpack(res[key + "4_codes"]), codes), key
        assert np.array_equal(res[key + "4_scales"], sbytes), key
    # the E4M3 token-block operands of the other products
    for key in ("q", "k", "v"):
        codes, sbytes, _ = OB.quantize_token_blocks(x[key], w.cu_seqlens)
        assert np.array_equal(res[key + "_codes"], codes), key
        assert np.array_equal(res[key + "_scales"], sbytes), key
    m = OB.in_doc_mask(w.cu_seqlens, w.T)
    f = OS.forward(x["q"], x["k"], x["v"], w.cu_seqlens, causal=causal, scores="nvfp4")
    assert np.isfinite(res["out"][m]).all() and np.isfinite(res["lse"][:, m]).all()
    e_o = rel_fro(res["out"][m], f["O"][m])
    e_l = rel_fro(res["lse"][:, m], f["lse"][:, m])
    assert e_o <= FWD_TOL and e_l <= FWD_TOL, (e_o, e_l)
    assert np.all(res["out"][~m] == 0) and np.all(np.isinf(res["lse"][:, ~m]))
    b = OS.backward(x["q"], x["k"], x["v"], f["O_bf16"], f["lse"], x["do"], w.cu_seqlens, causal=causal,
                    scores="nvfp4")
    errs = {}
    for key in ("dq", "dk", "dv"):
        assert np.isfinite(res[key]).all(), key
        errs[key] = rel_fro(res[key][m], b[key][m])
        assert errs[key] <= BWD_TOL, (key, errs[key])
        assert np.all(res[key][~m] == 0), key
    Ox, _ = OX.forward(x["q"], x["k"], x["v"], w.cu_seqlens, causal=causal)
    gx = OX.backward(x["q"], x["k"], x["v"], x["do"], w.cu_seqlens, causal=causal)
    print(f"\n{name} causal={causal}: vs oracle O {e_o:.2e} lse {e_l:.2e} {errs}; cosine to exact "
          f"(gpu, oracle): O ({cosine(res['out'][m], Ox[m]):.5f}, {cosine(f['O'][m], Ox[m]):.5f}) "
          f"dq ({cosine(res['dq'][m], gx[0][m]):.5f}, {cosine(b['dq'][m], gx[0][m]):.5f})")
