"""Parity at the full sizes of the benchmark workloads, in the launch configuration
bench.py times (persistent grid of one CTA per SM, many items per CTA).

The quantizer is checked bit-exactly over every token and head.  Attention
outputs are checked against the oracle on what it can compute in seconds: one
grouped-query group over all documents (d = 64 workload), sampled query tiles,
single heads, or document subsets (documents are independent, so the oracle on
a subset of documents gives exactly those rows).
"""
import numpy as np
import pytest

import workloads as W
from oracle import blocks as OB
from oracle import simulated as OS
from oracle import exact as OX
from tests.gpu_common import run_gpu, np_inputs, rel_fro, cosine

pytestmark = pytest.mark.gpu

FWD_TOL = 1e-2
BWD_TOL = 3e-2


def _codes_bit_exact(w, res, x):
    m = OB.in_doc_mask(w.cu_seqlens, w.T)
    for key, H in (("q", w.Hq), ("k", w.Hkv), ("v", w.Hkv)):
        codes, sb, _ = OB.quantize_token_blocks(x[key], w.cu_seqlens)
        assert np.array_equal(res[key + "_codes"][m], codes[m]), key
        assert np.array_equal(res[key + "_scales"][:, m], sb[:, m]), key
    codes, sb, _ = OB.quantize_token_blocks(x["do"], w.cu_seqlens)
    assert np.array_equal(res["do_codes"][m], codes[m]) and np.array_equal(res["do_scales"][:, m], sb[:, m])


def _sub_cu(cu, docs):
    """cu_seqlens restricted to some documents (absolute token offsets kept as separate documents)."""
    out = []
    for r in docs:
        out.append((int(cu[r]), int(cu[r + 1])))
    return out


def _check_docs(w, res, x, docs, heads, check_bwd=True, opts=None):
    """Oracle fwd (+bwd) on a subset of documents and heads of one KV group.

    Also reports the error against exact fp64 attention (cosine, as the pages'
    Section 4.2 does): the CUDA path must be as close to exact attention as the
    quantization-simulating oracle is, within 1e-3 of its cosine."""
    g = w.Hq // w.Hkv
    hk = heads[0] // g
    assert all(h // g == hk for h in heads)
    rows = np.concatenate([np.arange(s, e) for s, e in _sub_cu(w.cu_seqlens, docs)])
    # compact the chosen documents into their own packed sequence
    lens = [int(w.cu_seqlens[r + 1] - w.cu_seqlens[r]) for r in docs]
    cu = W.cu_from_lengths(lens)
    q = x["q"][rows][:, heads]; do = x["do"][rows][:, heads]
    k = x["k"][rows][:, [hk]]; v = x["v"][rows][:, [hk]]
    fwd_kw = dict(opts or {})
    bwd_kw = {kk: vv for kk, vv in fwd_kw.items() if kk != "v_fold"}   # the backward's dP takes per-key V
    f = OS.forward(q, k, v, cu, **fwd_kw)
    e_o = rel_fro(res["out"][rows][:, heads], f["O"])
    e_l = rel_fro(res["lse"][heads][:, rows], f["lse"])
    assert e_o <= FWD_TOL and e_l <= FWD_TOL, (e_o, e_l)
    out = {"O": e_o, "lse": e_l}
    if check_bwd:
        b = OS.backward(q, k, v, f["O_bf16"], f["lse"], do, cu, **bwd_kw)
        out["dq"] = rel_fro(res["dq"][rows][:, heads], b["dq"])
        if len(heads) == g:           # dK, dV sum over the whole group
            out["dk"] = rel_fro(res["dk"][rows][:, [hk]], b["dk"])
            out["dv"] = rel_fro(res["dv"][rows][:, [hk]], b["dv"])
        for kk in ("dq", "dk", "dv"):
            if kk in out:
                assert out[kk] <= BWD_TOL, (kk, out[kk])
    # against exact fp64 attention
    Ox, _ = OX.forward(q, k, v, cu)
    cos = {"O": (cosine(res["out"][rows][:, heads], Ox), cosine(f["O"], Ox))}
    if check_bwd:
        gx = OX.backward(q, k, v, do, cu)
        cos["dq"] = (cosine(res["dq"][rows][:, heads], gx[0]), cosine(b["dq"], gx[0]))
        if len(heads) == g:
            cos["dk"] = (cosine(res["dk"][rows][:, [hk]], gx[1]), cosine(b["dk"], gx[1]))
            cos["dv"] = (cosine(res["dv"][rows][:, [hk]], gx[2]), cosine(b["dv"], gx[2]))
    for kk, (c_gpu, c_orc) in cos.items():
        assert c_gpu >= c_orc - 1e-3, (kk, c_gpu, c_orc)
    out["cos_vs_exact(gpu, oracle)"] = {kk: (round(a, 5), round(b_, 5)) for kk, (a, b_) in cos.items()}
    return out


def _basic(w, res):
    m = OB.in_doc_mask(w.cu_seqlens, w.T)
    assert res["status"] == 0
    for key in ("out", "dq", "dk", "dv"):
        assert np.isfinite(res[key]).all(), key
    assert np.isfinite(res["lse"][:, m]).all()


def test_llama1b_packed_full():
    w = W.llama1b_packed()
    res = run_gpu(w)
    _basic(w, res)
    x = np_inputs(w)
    _codes_bit_exact(w, res, x)
    docs = list(range(w.n_docs))
    e = _check_docs(w, res, x, docs, heads=[0, 1, 2, 3])
    e2 = _check_docs(w, res, x, docs, heads=[28, 29, 30, 31], check_bwd=False)
    print(f"\nllama1b_packed group 0: {e}; group 7 fwd: {e2}")


def test_long_single_full():
    w = W.long_single()
    res = run_gpu(w)
    _basic(w, res)
    x = np_inputs(w)
    _codes_bit_exact(w, res, x)
    # one head, every query tile, forward and backward (MHA: the head is its own group)
    e = _check_docs(w, res, x, [0], heads=[5])
    print(f"\nlong_single head 5: {e}")


def test_skewed_full():
    w = W.skewed()
    res = run_gpu(w)
    _basic(w, res)
    x = np_inputs(w)
    _codes_bit_exact(w, res, x)
    L = np.diff(w.cu_seqlens)
    short = [r for r in range(w.n_docs) if L[r] <= 512][:40]
    e = _check_docs(w, res, x, short, heads=[4, 5, 6, 7])        # a whole group on the short documents
    longd = [r for r in range(w.n_docs) if L[r] == 16384][:1]
    e2 = _check_docs(w, res, x, longd, heads=[9], check_bwd=False)
    print(f"\nskewed short docs group 1: {e}; long doc head 9 fwd: {e2}")


def test_outliers_full():
    """Outlier channels (x20) push scores to tens of nats, where the E4M3 element error
    (up to 1/16) moves scores by several nats: the quantized computation itself is far
    from exact attention (the oracle's O differs from exact fp64 by ~30 %, its dK by
    ~100 %).  dK is then dominated by rounding-tie decisions, so on this workload it is
    held to equal accuracy against exact attention rather than to the 3e-2 distance
    from the oracle; O, LSE, dQ and dV keep the stated tolerances."""
    from oracle import exact as OX
    w = W.outliers()
    res = run_gpu(w)
    _basic(w, res)
    x = np_inputs(w)
    _codes_bit_exact(w, res, x)
    L = np.diff(w.cu_seqlens)
    docs = [r for r in range(w.n_docs) if L[r] <= 4096][:6]
    rows = np.concatenate([np.arange(w.cu_seqlens[r], w.cu_seqlens[r + 1]) for r in docs])
    cu = W.cu_from_lengths([int(L[r]) for r in docs])
    h = 3
    q, k, v, do = (x[n][rows][:, [h]] for n in ("q", "k", "v", "do"))
    f = OS.forward(q, k, v, cu)
    b = OS.backward(q, k, v, f["O_bf16"], f["lse"], do, cu)
    gpu = {"O": res["out"][rows][:, [h]], "dq": res["dq"][rows][:, [h]], "dk": res["dk"][rows][:, [h]],
           "dv": res["dv"][rows][:, [h]]}
    sim = {"O": f["O"], "dq": b["dq"], "dk": b["dk"], "dv": b["dv"]}
    assert rel_fro(res["lse"][h, rows], f["lse"][0]) <= FWD_TOL
    assert rel_fro(gpu["O"], sim["O"]) <= FWD_TOL
    for kk in ("dq", "dv"):
        assert rel_fro(gpu[kk], sim[kk]) <= BWD_TOL, kk
    Ox, _ = OX.forward(q, k, v, cu)
    gx = OX.backward(q, k, v, do, cu)
    e_gpu = rel_fro(gpu["dk"], gx[1])
    e_sim = rel_fro(sim["dk"], gx[1])
    assert abs(e_gpu - e_sim) <= 1e-2 * max(1.0, e_sim), (e_gpu, e_sim)
    print(f"\noutliers head {h}: dK vs oracle {rel_fro(gpu['dk'], sim['dk']):.3e}; vs exact: gpu {e_gpu:.3e}, "
          f"oracle {e_sim:.3e}; O vs exact: gpu {rel_fro(gpu['O'], Ox):.3e} oracle {rel_fro(sim['O'], Ox):.3e}")


def _unpack4(packed):
    lo = packed & 0xF
    hi = packed >> 4
    return np.stack([lo, hi], axis=-1).reshape(*packed.shape[:-1], packed.shape[-1] * 2)


def test_llama1b_packed_full_exact_options():
    """The exact options at the benchmark size: per-token codes and scales of
    Q, K, V, dO and the token-block V copy bit-exact over every token; one
    grouped-query group over all documents against the oracle with the same
    options (V folded on the diagonal tile in the forward)."""
    w = W.llama1b_packed()
    res = run_gpu(w, exact=True)
    _basic(w, res)
    x = np_inputs(w)
    m = OB.in_doc_mask(w.cu_seqlens, w.T)
    for key in ("q", "k", "v"):
        codes, sb, _ = OB.quantize_per_token(x[key], w.cu_seqlens)
        assert np.array_equal(res[key + "_codes"][m], codes[m]), key
        assert np.array_equal(res[key + "_scales"][:, m], sb[:, m]), key
    codes, sb, _ = OB.quantize_per_token(x["do"], w.cu_seqlens)
    assert np.array_equal(res["do_codes"][m], codes[m]) and np.array_equal(res["do_scales"][:, m], sb[:, m])
    codes, sb, _ = OB.quantize_token_blocks(x["v"], w.cu_seqlens)
    assert np.array_equal(res["vb_codes"][m], codes[m]) and np.array_equal(res["vb_scales"][:, m], sb[:, m])
    e = _check_docs(w, res, x, list(range(w.n_docs)), heads=[0, 1, 2, 3],
                    opts={"exact": True, "v_fold": "diagonal"})
    print(f"\nllama1b_packed exact options, group 0: {e}")


def test_llama1b_packed_full_nvfp4():
    """The mixed NVFP4/FP8 path at the benchmark size: NVFP4 Q and K codes and
    scales bit-exact over every token; one grouped-query group over all
    documents against the NVFP4 oracle."""
    from oracle import nvfp4 as ON
    w = W.llama1b_packed()
    res = run_gpu(w, nvfp4=True)
    _basic(w, res)
    x = np_inputs(w)
    m = OB.in_doc_mask(w.cu_seqlens, w.T)
    for key in ("q", "k"):
        codes, sb, _ = ON.quantize_nvfp4(x[key], w.cu_seqlens)
        assert np.array_equal(_unpack4(res[key + "4_codes"])[m], codes[m]), key
        assert np.array_equal(res[key + "4_scales"][m], sb[m]), key
    e = _check_docs(w, res, x, list(range(w.n_docs)), heads=[0, 1, 2, 3], opts={"scores": "nvfp4"})
    print(f"\nllama1b_packed NVFP4 path, group 0: {e}")


def test_llama1b_packed_full_deterministic_dq():
    """Order-independent dQ at the benchmark size: two runs give bitwise the
    same dQ, which agrees with the fp32 reduce-add path to 1e-3."""
    w = W.llama1b_packed()
    a = run_gpu(w, deterministic_dq=True)
    b = run_gpu(w, deterministic_dq=True)
    ref = run_gpu(w)
    for r in (a, b, ref):
        _basic(w, r)
    assert np.array_equal(a["dq"], b["dq"])
    for key in ("out", "lse", "dk", "dv"):
        assert np.array_equal(a[key], ref[key]), key
    m = OB.in_doc_mask(w.cu_seqlens, w.T)
    assert rel_fro(a["dq"][m], ref["dq"][m]) < 1e-3
