"""The order-independent dQ option (flamia_opts.deterministic_dq) on the GPU.

Each dQ partial (one per key tile, query row and channel) is added as a 64-bit
fixed-point integer, so the accumulated dQ does not depend on the order in
which key tiles finish.  These tests check that dQ is then bitwise
reproducible (across runs and work hand-outs), that it stays within the
backward tolerance of the quantization-simulating oracle, and that documents
of several key tiles leak nothing into one another, bit for bit (FLAMIA
Appendix B.5 on deterministic reductions; the spec bar of zero
cross-document leakage).
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import blocks as OB
from oracle import simulated as OS
from tests.gpu_common import run_gpu, np_inputs, rel_fro

pytestmark = pytest.mark.gpu

BWD_TOL = 3e-2


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_deterministic_dq_parity_and_reproducibility(d, causal):
    # documents of several key tiles, a ragged tail and padding rows
    w = W.custom([700, 17, 300, 0, 430], Hq=4, Hkv=2, d=d, seed=31, T=1500)
    runs = [run_gpu(w, causal=causal, deterministic_dq=True),
            run_gpu(w, causal=causal, deterministic_dq=True),
            run_gpu(w, causal=causal, deterministic_dq=True, schedule="static")]
    for r in runs:
        assert r["status"] == 0
    for r in runs[1:]:
        for key in ("out", "lse", "dq", "dk", "dv"):
            assert np.array_equal(runs[0][key], r[key]), key
    res = runs[0]
    x = np_inputs(w)
    m = OB.in_doc_mask(w.cu_seqlens, w.T)
    f = OS.forward(x["q"], x["k"], x["v"], w.cu_seqlens, causal=causal)
    b = OS.backward(x["q"], x["k"], x["v"], f["O_bf16"], f["lse"], x["do"], w.cu_seqlens, causal=causal)
    for key in ("dq", "dk", "dv"):
        assert np.isfinite(res[key]).all(), key
        e = rel_fro(res[key][m], b[key][m])
        assert e <= BWD_TOL, (key, e)
        assert np.all(res[key][~m] == 0), key
    # the fp32 path computes the same sums up to rounding
    ref = run_gpu(w, causal=causal)
    assert rel_fro(res["dq"][m], ref["dq"][m]) < 1e-3
    for key in ("out", "lse", "dk", "dv"):
        assert np.array_equal(res[key], ref[key]), key


@pytest.mark.parametrize("d", [64, 128])
def test_cross_document_leakage_long_documents_bitwise(d):
    # documents of several key tiles: with the deterministic option every output,
    # dQ included, is bitwise independent of another document's contents
    w = W.custom([700, 300, 500], Hq=2, Hkv=1, d=d, seed=7)
    base = run_gpu(w, deterministic_dq=True)
    t2 = {n: w.tensors[n].clone() for n in w.tensors}
    s, e = int(w.cu_seqlens[1]), int(w.cu_seqlens[2])
    for n in t2:
        t2[n][s:e] = (t2[n][s:e].float() * 1e4).to(torch.bfloat16)
    pert = run_gpu(w, tensors=t2, deterministic_dq=True)
    assert base["status"] == 0 and pert["status"] == 0
    keep = np.ones(w.T, bool); keep[s:e] = False
    for key in ("out", "dq", "dk", "dv"):
        assert np.array_equal(base[key][keep], pert[key][keep]), key
    assert np.array_equal(base["lse"][:, keep], pert["lse"][:, keep])
    assert not np.array_equal(base["dq"][s:e], pert["dq"][s:e])


@pytest.mark.parametrize("d", [64, 128])
def test_exact_options_future_token_dq_bitwise_across_key_tiles(d):
    """Exact options with the deterministic option: a later token of a
    five-tile document scaled by 2^12 in Q, K, V and dO changes no bit of any
    earlier row's dQ, although those rows sum partials from several key
    tiles (without the option only rows within one key tile can be compared
    bitwise)."""
    w = W.custom([600, 200], Hq=2, Hkv=1, d=d, seed=23, T=820)
    tp = 470
    base = {n: w.tensors[n].clone() for n in w.tensors}
    pert = {n: w.tensors[n].clone() for n in w.tensors}
    for n in ("q", "k", "v", "do"):
        pert[n][tp] = (pert[n][tp].float() * 4096.0).to(torch.bfloat16)
    r0 = run_gpu(w, tensors=base, exact=True, deterministic_dq=True)
    r1 = run_gpu(w, tensors=pert, exact=True, deterministic_dq=True)
    assert r0["status"] == 0 and r1["status"] == 0
    assert np.array_equal(r0["dq"][:tp], r1["dq"][:tp])
    assert np.array_equal(r0["out"][:tp], r1["out"][:tp])
    assert np.array_equal(r0["dq"][600:], r1["dq"][600:])          # the other document
    assert not np.array_equal(r0["dq"][tp:600], r1["dq"][tp:600])
