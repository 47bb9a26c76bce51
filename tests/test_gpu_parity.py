"""GPU parity of the CUDA path against the CPU oracle (run through the C-ABI).

Bar (from the method's acceptance criteria): quantized codes and scales of Q, K,
V and dO bit-exact; relative Frobenius error <= 1e-2 for O and LSE and <= 3e-2
for dQ, dK, dV against the quantization-simulating oracle; cross-document
leakage exactly zero.  Errors against exact fp64 attention are reported.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import blocks as OB
from oracle import exact as OX
from oracle import hadamard as OH
from oracle import simulated as OS
from tests.gpu_common import run_gpu, np_inputs, rel_fro, cosine
import precision_causal_attention_gb300 as F

pytestmark = pytest.mark.gpu

FWD_TOL = 1e-2
BWD_TOL = 3e-2


def _in_doc(w):
    return OB.in_doc_mask(w.cu_seqlens, w.T)


def _check_codes(w, res, x, key, H):
    # every token, including those outside documents (code 0, scale byte 0 on both sides)
    codes, sbytes, _ = OB.quantize_token_blocks(x, w.cu_seqlens)
    assert np.array_equal(res[key + "_codes"], codes), key
    assert np.array_equal(res[key + "_scales"], sbytes), key


SMALL = [
    ("tiny", lambda: W.tiny()),
    ("ragged_d64_gqa", lambda: W.custom([300, 17, 129, 0, 256, 1, 40], Hq=4, Hkv=2, d=64, seed=3, T=800)),
    ("ragged_d128", lambda: W.custom([260, 128, 33, 400], Hq=2, Hkv=1, d=128, seed=4, T=840)),
    # fixed-length batch (one document per sequence, no packing)
    ("batched_d64", lambda: W.custom([384, 384, 384], Hq=4, Hkv=1, d=64, seed=6, T=1152)),
]


@pytest.mark.parametrize("name,make", SMALL, ids=[s[0] for s in SMALL])
@pytest.mark.parametrize("causal", [True, False])
def test_small_parity(name, make, causal):
    w = make()
    res = run_gpu(w, causal=causal)
    assert res["status"] == 0
    x = np_inputs(w)
    # operand codes and scales, bit-exact
    _check_codes(w, res, x["q"], "q", w.Hq)
    _check_codes(w, res, x["k"], "k", w.Hkv)
    _check_codes(w, res, x["v"], "v", w.Hkv)
    f = OS.forward(x["q"], x["k"], x["v"], w.cu_seqlens, causal=causal)
    m = _in_doc(w)
    assert np.isfinite(res["out"][m]).all() and np.isfinite(res["lse"][:, m]).all()
    e_o = rel_fro(res["out"][m], f["O"][m])
    e_l = rel_fro(res["lse"][:, m], f["lse"][:, m])
    assert e_o <= FWD_TOL and e_l <= FWD_TOL, (e_o, e_l)
    # rows outside documents
    assert np.all(res["out"][~m] == 0) and np.all(np.isinf(res["lse"][:, ~m]))
    # backward
    b = OS.backward(x["q"], x["k"], x["v"], f["O_bf16"], f["lse"], x["do"], w.cu_seqlens, causal=causal)
    (doh, doc_, dos, _), D = b["do"], b["D"]
    assert np.array_equal(res["do_codes"], doc_) and np.array_equal(res["do_scales"], dos)
    # D derives from O, which matches only within the forward tolerance
    assert rel_fro(res["D"][:, m], D[:, m]) < FWD_TOL
    for key in ("dq", "dk", "dv"):
        assert np.isfinite(res[key]).all(), key
        e = rel_fro(res[key][m], b[key][m])
        assert e <= BWD_TOL, (key, e)
        assert np.all(res[key][~m] == 0), key
    # exact fp64 attention, reported
    Ox, _ = OX.forward(x["q"], x["k"], x["v"], w.cu_seqlens, causal=causal)
    gx = OX.backward(x["q"], x["k"], x["v"], x["do"], w.cu_seqlens, causal=causal)
    print(f"\n{name} causal={causal}: vs simulated O {e_o:.2e}; vs exact O cos {cosine(res['out'][m], Ox[m]):.5f} "
          f"dq cos {cosine(res['dq'][m], gx[0][m]):.5f} dk cos {cosine(res['dk'][m], gx[1][m]):.5f} "
          f"dv cos {cosine(res['dv'][m], gx[2][m]):.5f}")


def test_forward_is_bitwise_deterministic():
    w = W.custom([500, 300], Hq=4, Hkv=1, d=64, seed=5)
    a = run_gpu(w, do_bwd=False)
    b = run_gpu(w, do_bwd=False)
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["lse"], b["lse"])


@pytest.mark.parametrize("d", [64, 128])
def test_cross_document_leakage_is_exactly_zero(d):
    # documents of <= 128 tokens: each dQ element receives exactly one atomic add,
    # so every output is deterministic and the comparison can be bitwise
    lengths = [100, 128, 77, 128, 5]
    w = W.custom(lengths, Hq=4, Hkv=2, d=d, seed=6)
    base = run_gpu(w)
    t2 = {n: w.tensors[n].clone() for n in w.tensors}
    s, e = int(w.cu_seqlens[1]), int(w.cu_seqlens[2])
    for n in t2:
        t2[n][s:e] = (t2[n][s:e].float() * 1e4).to(torch.bfloat16)
    pert = run_gpu(w, tensors=t2)
    keep = np.ones(w.T, bool); keep[s:e] = False
    for key in ("out", "dq", "dk", "dv"):
        assert np.array_equal(base[key][keep], pert[key][keep]), key
    assert np.array_equal(base["lse"][:, keep], pert["lse"][:, keep])
    assert not np.array_equal(base["out"][s:e], pert["out"][s:e])


def test_cross_document_leakage_long_documents_dk_dv():
    # long documents: dK, dV (accumulated in tensor memory, written once) are bitwise
    # reproducible; dQ uses atomics and is compared within rounding
    w = W.custom([700, 300, 500], Hq=2, Hkv=1, d=64, seed=7)
    base = run_gpu(w)
    t2 = {n: w.tensors[n].clone() for n in w.tensors}
    s, e = int(w.cu_seqlens[1]), int(w.cu_seqlens[2])
    for n in t2:
        t2[n][s:e] = (t2[n][s:e].float() * 1e4).to(torch.bfloat16)
    pert = run_gpu(w, tensors=t2)
    keep = np.ones(w.T, bool); keep[s:e] = False
    for key in ("out", "dk", "dv"):
        assert np.array_equal(base[key][keep], pert[key][keep]), key
    assert rel_fro(pert["dq"][keep], base["dq"][keep]) < 1e-5


def test_bad_cu_seqlens_reported_on_device():
    w = W.custom([64, 64], Hq=2, Hkv=2, d=64, seed=8)
    w.cu_seqlens = np.array([0, 100, 90], np.int32)       # decreasing
    res = run_gpu(w, do_bwd=False)
    assert res["status"] == 1


@pytest.mark.parametrize("d", [64, 128])
def test_cuda_graph_replay_matches_eager(d):
    """The fwd+bwd calls allocate nothing and never synchronise, so a whole step
    can be captured into one CUDA graph; replays (after the inputs change in
    place) give the eager results: forward outputs, dK and dV bitwise (fixed
    accumulation order), dQ up to the order of the fp32 reduce-adds."""
    w = W.custom([500, 300, 77], Hq=4, Hkv=2, d=d, seed=11, T=900)
    dev = torch.device("cuda:0")
    q, k, v, do = (w.tensors[n].to(dev) for n in ("q", "k", "v", "do"))
    cu = torch.from_numpy(np.asarray(w.cu_seqlens, np.int32)).to(dev)
    B = F.Buffers(w.T, w.n_docs, w.Hq, w.Hkv, d)
    opts = F.default_opts()

    def step():
        F.flamia_fwd(q, k, v, cu, B.out, B.lse, B.saved, B.work, opts)
        F.flamia_bwd(B.out, B.lse, do, cu, B.saved, B.dq, B.dk, B.dv, B.work, opts)

    def snapshot():
        torch.cuda.synchronize()
        return {n: getattr(B, n).clone() for n in ("out", "lse", "dq", "dk", "dv")}

    step()
    snapshot()                                        # first-use set-up happens outside capture
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    gen = torch.Generator().manual_seed(12)
    for _ in range(2):
        for t in (q, k, v, do):                       # new inputs, same buffers
            t.copy_(torch.randn(t.shape, generator=gen).to(torch.bfloat16))
        step()
        eager = snapshot()
        g.replay()
        replay = snapshot()
        assert F.flamia_get_status() == 0
        for n in ("out", "lse", "dk", "dv"):
            assert torch.equal(eager[n], replay[n]), n
        # bf16 rounding of an fp32 sum taken in another order may move an element by one ulp
        assert rel_fro(replay["dq"].float().cpu().numpy(), eager["dq"].float().cpu().numpy()) < 2e-3


def test_dq_accumulator_zeroing_paths():
    """The forward zeroes the dQ accumulator of its workspace and stamps it; the
    backward then skips the zeroing.  A backward on a workspace that was not
    stamped (a second backward, or a workspace full of garbage) must zero it
    itself and give the same gradients."""
    w = W.custom([700, 300, 61], Hq=4, Hkv=2, d=64, seed=13, T=1100)
    dev = torch.device("cuda:0")
    q, k, v, do = (w.tensors[n].to(dev) for n in ("q", "k", "v", "do"))
    cu = torch.from_numpy(np.asarray(w.cu_seqlens, np.int32)).to(dev)
    B = F.Buffers(w.T, w.n_docs, w.Hq, w.Hkv, w.d)
    opts = F.default_opts()

    def grads():
        torch.cuda.synchronize()
        return [x.float().cpu().numpy() for x in (B.dq, B.dk, B.dv)]

    F.flamia_fwd(q, k, v, cu, B.out, B.lse, B.saved, B.work, opts)
    F.flamia_bwd(B.out, B.lse, do, cu, B.saved, B.dq, B.dk, B.dv, B.work, opts)
    ref = grads()
    # second backward: the stamp was consumed, the accumulator holds the last sums
    F.flamia_bwd(B.out, B.lse, do, cu, B.saved, B.dq, B.dk, B.dv, B.work, opts)
    again = grads()
    # a workspace that never saw a forward, filled with garbage
    B.work.fill_(0xFF)
    F.flamia_bwd(B.out, B.lse, do, cu, B.saved, B.dq, B.dk, B.dv, B.work, opts)
    fresh = grads()
    assert F.flamia_get_status() == 0
    for a_, b_, c_ in zip(ref, again, fresh):
        assert rel_fro(b_, a_) < 2e-3 and rel_fro(c_, a_) < 2e-3
    assert np.array_equal(ref[1], fresh[1]) and np.array_equal(ref[2], fresh[2])


def test_host_pipeline_matches_direct_calls():
    """Batches in pinned host memory run through HostPipeline (copies on their
    own streams, two batches in flight, two device slots) give the results of
    direct calls on the same inputs: out, lse, dK, dV bitwise, dQ up to the
    order of the fp32 reduce-adds.  Consecutive batches differ in inputs and
    in their document lengths."""
    from precision_causal_attention_gb300.host_pipeline import HostPipeline
    ws = [W.custom([500, 300, 77], Hq=4, Hkv=2, d=64, seed=21, T=900),
          W.custom([128, 640, 90, 20], Hq=4, Hkv=2, d=64, seed=22, T=900),
          W.custom([899], Hq=4, Hkv=2, d=64, seed=23, T=900)]
    dev = torch.device("cuda:0")
    opts = F.default_opts()
    max_docs = max(w.n_docs for w in ws)
    pipe = HostPipeline(900, max_docs, 4, 2, 64, device=dev, opts=opts)
    names = ("out", "lse", "dq", "dk", "dv")
    hins, houts, refs = [], [], []
    for w in ws:
        hin = {n: w.tensors[n].pin_memory() for n in ("q", "k", "v", "do")}
        hin["cu"] = torch.from_numpy(np.asarray(w.cu_seqlens, np.int32)).pin_memory()
        B = F.Buffers(w.T, w.n_docs, w.Hq, w.Hkv, w.d)
        houts.append({n: torch.empty(getattr(B, n).shape, dtype=getattr(B, n).dtype).pin_memory() for n in names})
        hins.append(hin)
        q, k, v, do = (w.tensors[n].to(dev) for n in ("q", "k", "v", "do"))
        cu = torch.from_numpy(np.asarray(w.cu_seqlens, np.int32)).to(dev)
        F.flamia_fwd(q, k, v, cu, B.out, B.lse, B.saved, B.work, opts)
        F.flamia_bwd(B.out, B.lse, do, cu, B.saved, B.dq, B.dk, B.dv, B.work, opts)
        torch.cuda.synchronize()
        refs.append({n: getattr(B, n).cpu() for n in names})
    for i in range(2):                                  # each batch twice, so both slots get reused
        for hin, hout in zip(hins, houts):
            pipe.submit(hin, hout)
        pipe.synchronize()
        assert F.flamia_get_status() == 0
        for hout, ref in zip(houts, refs):
            for n in ("out", "lse", "dk", "dv"):
                assert torch.equal(hout[n], ref[n]), n
            assert rel_fro(hout["dq"].float().numpy(), ref["dq"].float().numpy()) < 2e-3
    h2d, d2h = HostPipeline.bytes_per_batch(hins[0], houts[0])
    assert h2d == (900 * 4 * 64 * 2) * 2 + (900 * 2 * 64 * 2) * 2 + 4 * 4
    assert d2h == 900 * 4 * 64 * 2 * 2 + 4 * 900 * 4 + 900 * 2 * 64 * 2 * 2


@pytest.mark.parametrize("causal", [True, False])
def test_hadamard_rotation_d128_parity(causal):
    """Hadamard option (d = 128): Q and K are rotated in fp32 before quantization;
    their codes and scales equal the oracle's codes of the rotated values bit for
    bit, and O, LSE, dQ, dK, dV (mapped back) match the rotated oracle."""
    w = W.custom([260, 128, 33, 400], Hq=2, Hkv=1, d=128, seed=14, T=840)
    t = {n: w.tensors[n].clone() for n in w.tensors}
    for n in ("q", "k"):                            # a few outlier channels, as the rotation is meant for
        x = t[n].float()
        x[:, :, 5] *= 20.0
        x[:, :, 77] *= 12.0
        t[n] = x.to(torch.bfloat16)
    res = run_gpu(w, causal=causal, tensors=t, hadamard=True)
    assert res["status"] == 0
    x = np_inputs(w, t)
    _check_codes(w, res, OH.rotate(x["q"]), "q", w.Hq)
    _check_codes(w, res, OH.rotate(x["k"]), "k", w.Hkv)
    _check_codes(w, res, x["v"], "v", w.Hkv)
    f = OS.forward(x["q"], x["k"], x["v"], w.cu_seqlens, causal=causal, hadamard=True)
    m = _in_doc(w)
    e_o = rel_fro(res["out"][m], f["O"][m])
    e_l = rel_fro(res["lse"][:, m], f["lse"][:, m])
    assert e_o <= FWD_TOL and e_l <= FWD_TOL, (e_o, e_l)
    b = OS.backward(x["q"], x["k"], x["v"], f["O_bf16"], f["lse"], x["do"], w.cu_seqlens, causal=causal,
                    hadamard=True)
    for key in ("dq", "dk", "dv"):
        e = rel_fro(res[key][m], b[key][m])
        assert e <= BWD_TOL, (key, e)
        assert np.all(res[key][~m] == 0), key
    # the rotation leaves the scores unchanged: against exact attention the
    # rotated path is as close as the plain one
    Ox, _ = OX.forward(x["q"], x["k"], x["v"], w.cu_seqlens, causal=causal)
    assert cosine(res["out"][m], Ox[m]) > 0.99


EXACT = [
    ("ragged_d64_gqa", lambda: W.custom([300, 17, 129, 0, 256, 1, 40], Hq=4, Hkv=2, d=64, seed=17, T=800)),
    ("ragged_d128", lambda: W.custom([260, 128, 33, 400], Hq=2, Hkv=1, d=128, seed=18, T=840)),
]


@pytest.mark.parametrize("name,make", EXACT, ids=[s[0] for s in EXACT])
@pytest.mark.parametrize("causal", [True, False])
def test_exact_options_forward_parity(name, make, causal):
    """Exact options (forward): per-token Q, K, V codes and scales and the
    token-block V copy bit-exact against the oracle's quantizers; O and LSE
    within the forward tolerance of the oracle with the same options (V's
    per-key exponents folded into P-hat on the diagonal tile of a causal call,
    token-block V on the tiles before it, as FLAMIA Section 3.2 does)."""
    w = make()
    t = {n: w.tensors[n].clone() for n in w.tensors}
    for n in ("q", "k", "v"):                       # token magnitudes spread over 2^-6 .. 2^6
        g = torch.Generator().manual_seed(5 + len(n))
        f = torch.exp2(torch.randint(-6, 7, (w.T, 1, 1), generator=g).float())
        t[n] = (t[n].float() * f).to(torch.bfloat16)
    res = run_gpu(w, causal=causal, tensors=t, do_bwd=False, exact=True)
    assert res["status"] == 0
    x = np_inputs(w, t)
    for key in ("q", "k", "v"):
        codes, sbytes, _ = OB.quantize_per_token(x[key], w.cu_seqlens)
        assert np.array_equal(res[key + "_codes"], codes), key
        assert np.array_equal(res[key + "_scales"], sbytes), key
    codes, sbytes, _ = OB.quantize_token_blocks(x["v"], w.cu_seqlens)
    assert np.array_equal(res["vb_codes"], codes) and np.array_equal(res["vb_scales"], sbytes)
    f = OS.forward(x["q"], x["k"], x["v"], w.cu_seqlens, causal=causal, exact=True, v_fold="diagonal")
    m = _in_doc(w)
    assert np.isfinite(res["out"][m]).all() and np.isfinite(res["lse"][:, m]).all()
    e_o = rel_fro(res["out"][m], f["O"][m])
    e_l = rel_fro(res["lse"][:, m], f["lse"][:, m])
    assert e_o <= FWD_TOL and e_l <= FWD_TOL, (e_o, e_l)
    assert np.all(res["out"][~m] == 0) and np.all(np.isinf(res["lse"][:, ~m]))


@pytest.mark.parametrize("d,which", [(64, ("q", "k", "v")), (128, ("q", "k", "v")), (64, ("do",)),
                                     (128, ("do",)), (64, ("q", "k", "v", "do")), (128, ("q", "k", "v", "do"))])
def test_exact_options_future_token_changes_no_earlier_row(d, which):
    """A later token of the same 32-token block scaled by 2^12 in the given
    operands (every scale group holding it jumps) leaves every bit of the
    earlier rows' O, LSE and dQ (one key tile, so one reduce-add per row)
    unchanged with the exact options; with token-block scales the rows of
    its block before it move (the in-block residue)."""
    w = W.custom([300, 200], Hq=2, Hkv=1, d=d, seed=19, T=520)
    tp = 45
    bwd = True
    base = {n: w.tensors[n].clone() for n in w.tensors}
    pert = {n: w.tensors[n].clone() for n in w.tensors}
    for n in which:
        pert[n][tp] = (pert[n][tp].float() * 4096.0).to(torch.bfloat16)
    r0 = run_gpu(w, tensors=base, do_bwd=bwd, exact=True)
    r1 = run_gpu(w, tensors=pert, do_bwd=bwd, exact=True)
    assert r0["status"] == 0 and r1["status"] == 0
    assert np.array_equal(r0["out"][:tp], r1["out"][:tp])
    assert np.array_equal(r0["lse"][:, :tp], r1["lse"][:, :tp])
    assert np.array_equal(r0["out"][300:], r1["out"][300:])        # the other document
    if bwd:
        assert np.array_equal(r0["dq"][:tp], r1["dq"][:tp])
        for key in ("dk", "dv"):
            assert np.array_equal(r0[key][300:], r1[key][300:])
    d0 = run_gpu(w, tensors=base, do_bwd=bwd)
    d1 = run_gpu(w, tensors=pert, do_bwd=bwd)
    if which == ("do",):
        assert not np.array_equal(d0["dq"][32:tp], d1["dq"][32:tp])   # the 32 x 32 dS blocks
    else:
        assert not np.array_equal(r0["out"][tp:300], r1["out"][tp:300])
        assert not np.array_equal(d0["out"][32:tp], d1["out"][32:tp])


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_exact_options_backward_parity(causal, d):
    """Exact options (backward): per-token dO codes and scales bit-exact; dQ,
    dK, dV within the backward tolerance of the oracle with the same options
    (K-folded per-row dS for dQ, Q-folded 32 x 32 dS for dK, dO-folded P' for
    dV).  At d = 64 S and dP are block-scaled MMAs with K's and V's per-key
    scales; at d = 128 they are unscaled MMAs with per-column factors."""
    w = W.custom([300, 17, 129, 0, 256, 1, 40], Hq=4, Hkv=2, d=d, seed=20, T=800)
    t = {n: w.tensors[n].clone() for n in w.tensors}
    for n in ("q", "k", "v", "do"):                 # token magnitudes spread over 2^-6 .. 2^6
        g = torch.Generator().manual_seed(7 + len(n))
        f = torch.exp2(torch.randint(-6, 7, (w.T, 1, 1), generator=g).float())
        t[n] = (t[n].float() * f).to(torch.bfloat16)
    res = run_gpu(w, causal=causal, tensors=t, exact=True)
    assert res["status"] == 0
    x = np_inputs(w, t)
    codes, sbytes, _ = OB.quantize_per_token(x["do"], w.cu_seqlens)
    assert np.array_equal(res["do_codes"], codes) and np.array_equal(res["do_scales"], sbytes)
    m = _in_doc(w)
    # the forward folds V on the diagonal tile only; the backward's dP takes
    # V's per-key scales on every tile
    f = OS.forward(x["q"], x["k"], x["v"], w.cu_seqlens, causal=causal, exact=True, v_fold="diagonal")
    b = OS.backward(x["q"], x["k"], x["v"], f["O_bf16"], f["lse"], x["do"], w.cu_seqlens, causal=causal,
                    exact=True)
    for key in ("dq", "dk", "dv"):
        e = rel_fro(res[key][m], b[key][m])
        assert e <= BWD_TOL, (key, e)
        assert np.all(res[key][~m] == 0), key
