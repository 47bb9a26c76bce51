"""Pins for the exact options of the oracle (per-token operand scales, the V
fold into P-hat, the per-query-row dS exponent with the K fold): FLAMIA,
Section 3.2 (leak mechanism, folds of per-key scales), Section 4.5 (only the
exact options leave earlier outputs unchanged) and Appendix A.3 (the in-block
residue they close)."""
import numpy as np
import pytest

from oracle import blocks as B
from oracle import exact as X
from oracle import formats as F
from oracle import simulated as S


def _bf16_inputs(T, Hq, Hkv, d, seed=0):
    rng = np.random.default_rng(seed)
    f = lambda shp: F.bf16_round(rng.standard_normal(shp))
    return f((T, Hq, d)), f((T, Hkv, d)), f((T, Hkv, d)), f((T, Hq, d))


def _run(q, k, v, do, cu, exact, causal=True, v_fold="all"):
    f = S.forward(q, k, v, cu, causal=causal, exact=exact, v_fold=v_fold)
    b = S.backward(q, k, v, f["O_bf16"], f["lse"], do, cu, causal=causal, exact=exact, v_fold=v_fold)
    return f, b


def test_per_token_quantizer_is_the_block_quantizer_on_one_token_documents():
    rng = np.random.default_rng(0)
    x = F.bf16_round(rng.standard_normal((90, 3, 16)) * np.exp2(rng.integers(-20, 20, (90, 3, 1))))
    cu = [0, 37, 37, 90]
    c1, s1, e1 = B.quantize_per_token(x, cu)
    c2, s2, e2 = B.quantize_token_blocks(x, list(range(91)))
    assert np.array_equal(c1, c2) and np.array_equal(s1, s2) and np.array_equal(e1, e2)
    # and the exponent is the smallest admissible one, token by token
    amax = np.abs(x).max(axis=2).T
    assert np.all(amax <= 448.0 * np.exp2(e1.astype(float)))
    assert np.all(amax > 448.0 * np.exp2(e1.astype(float) - 1))


def test_row_dS_quantizer_is_the_32x32_quantizer_row_by_row():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((7, 77)) * np.exp2(rng.integers(-30, 5, (7, 77)))
    vals, codes, E = S.ds_quantize_rows(x)
    for r in range(7):
        v1, c1, e1 = S.ds_quantize(x[r:r + 1])
        assert np.array_equal(vals[r:r + 1], v1) and np.array_equal(codes[r:r + 1], c1)
        assert np.array_equal(E[r], e1[0])


def _uniform_block_exponents(x, seed):
    """Every token row gets the same maximum magnitude (1.5 times a per-32-token-
    block power of two), so its per-token exponent equals its block exponent."""
    rng = np.random.default_rng(seed)
    y = np.clip(x, -1.0, 1.0).copy()
    T = y.shape[0]
    for b0 in range(0, T, 32):
        y[b0:b0 + 32] *= 2.0 ** int(rng.integers(-6, 7))
        y[b0:b0 + 32, :, 0] = 1.5 * 2.0 ** int(rng.integers(-6, 7))
    return F.bf16_round(y)


@pytest.mark.parametrize("causal", [True, False])
def test_folds_reduce_to_the_default_path_when_exponents_are_block_uniform(causal):
    """With block-uniform exponents the per-token codes are the token-block
    codes, the V fold is 2^c, the Q fold shifts each 32 x 32 dS block
    exponent and the dO fold is 2^8: O, LSE, dK and dV equal the default path
    bit for bit.  A dropped or sign-flipped fold exponent breaks this."""
    cu = [0, 160]                                      # blocks of 32 start on document boundaries
    q, k, v, do = (_uniform_block_exponents(x, s) for s, x in enumerate(_bf16_inputs(160, 2, 1, 16, seed=3)))
    f0, b0 = _run(q, k, v, do, cu, exact=False, causal=causal)
    f1, b1 = _run(q, k, v, do, cu, exact=True, causal=causal)
    for n in ("q", "k", "v"):
        assert np.array_equal(f0[n][1], f1[n][1]) and np.array_equal(f0[n][3], f1[n][3])
    assert np.array_equal(f0["O"], f1["O"]) and np.array_equal(f0["lse"], f1["lse"])
    assert np.array_equal(b0["dk"], b1["dk"]) and np.array_equal(b0["dv"], b1["dv"])
    # dQ differs only through the row-wise dS exponents: same order of error
    gx = X.backward(q, k, v, do, cu, causal=causal)
    rel = lambda a, b: np.linalg.norm(a - b) / np.linalg.norm(b)
    assert rel(b1["dq"], gx[0]) < 2 * rel(b0["dq"], gx[0]) + 1e-3


def test_exact_options_stay_close_to_exact_attention():
    cu = [0, 200, 333, 600]
    q, k, v, do = _bf16_inputs(600, 4, 2, 32, seed=4)
    Ox, lx = X.forward(q, k, v, cu)
    gx = X.backward(q, k, v, do, cu)
    rel = lambda a, b: np.linalg.norm(a - b) / np.linalg.norm(b)
    f0, b0 = _run(q, k, v, do, cu, exact=False)
    f1, b1 = _run(q, k, v, do, cu, exact=True)
    assert rel(f1["O"], Ox) < 5e-2
    assert rel(f1["O"], Ox) < 1.5 * rel(f0["O"], Ox)
    assert f1["pmax"] <= 2.0 ** (4 + 4)                # the fold never raises the P-hat input
    for i, key in enumerate(("dq", "dk", "dv")):
        e1, e0 = rel(b1[key], gx[i]), rel(b0[key], gx[i])
        assert e1 < 1e-1 and e1 < 1.5 * e0 + 1e-3, (key, e1, e0)


def _future_perturbation(exact, which, t=45, L=150, v_fold="all"):
    """(forward, backward) before and after token t of a 150-token document is
    scaled by 2^12 in the operands ``which`` (every scale group holding t
    jumps; dO alone scales row t of dS)."""
    q, k, v, do = _bf16_inputs(L + 30, 2, 1, 16, seed=5)
    cu = [0, L, L + 30]
    a = _run(q, k, v, do, cu, exact, v_fold=v_fold)
    xs = {"q": q.copy(), "k": k.copy(), "v": v.copy(), "do": do.copy()}
    for n in which:
        xs[n][t] *= 4096.0
    b = _run(xs["q"], xs["k"], xs["v"], xs["do"], cu, exact, v_fold=v_fold)
    return a, b


WHICH = (("q",), ("k",), ("v",), ("do",), ("q", "k", "v", "do"))


@pytest.mark.parametrize("v_fold", ["all", "diagonal"])
@pytest.mark.parametrize("which", WHICH)
def test_exact_options_leave_earlier_rows_unchanged(which, v_fold):
    t = 45
    (fa, ba), (fb, bb) = _future_perturbation(True, which, t, v_fold=v_fold)
    assert np.array_equal(fa["O"][:t], fb["O"][:t])
    assert np.array_equal(fa["lse"][:, :t], fb["lse"][:, :t])
    assert np.array_equal(ba["dq"][:t], bb["dq"][:t])
    # the other document is untouched in every output
    for key in ("dq", "dk", "dv"):
        assert np.array_equal(ba[key][150:], bb[key][150:])
    assert np.array_equal(fa["O"][150:], fb["O"][150:])
    # and the perturbation is real: later rows or the gradients move
    assert any(not np.array_equal(x[t:150], y[t:150]) for x, y in
               ((fa["O"], fb["O"]), (ba["dq"], bb["dq"]), (ba["dk"], bb["dk"]), (ba["dv"], bb["dv"])))


@pytest.mark.parametrize("which", WHICH)
def test_default_scaling_leaks_inside_the_block_negative_control(which):
    """The same probes on the default token-block / 32 x 32 scaling move rows
    of t's block before t (the in-block residue of Appendix A.3)."""
    t = 45
    (fa, ba), (fb, bb) = _future_perturbation(False, which, t)
    blk = slice(32, t)                                 # rows of t's 32-token block before t
    moved = {n: not np.array_equal(x[blk], y[blk]) for n, (x, y) in
             {"O": (fa["O"], fb["O"]), "dq": (ba["dq"], bb["dq"])}.items()}
    assert moved["O"] or moved["dq"]
    if which == ("do",):
        assert moved["dq"]                             # through the 32 x 32 dS blocks only
    # rows of the first block read t only through scale groups they do not share
    assert np.array_equal(fa["O"][:32], fb["O"][:32])


def test_diagonal_only_v_fold():
    """The V fold restricted to the diagonal tile (Section 3.2): rows whose
    query tile has no earlier key tile see only the diagonal and match the
    all-tile fold bit for bit; later rows read block-coded V on the earlier
    tiles; the probes above also hold for a future token in a later tile."""
    q, k, v, do = _bf16_inputs(400, 2, 1, 32, seed=11)
    cu = [0, 300, 400]
    fa, ba = _run(q, k, v, do, cu, True, v_fold="all")
    fd, bd = _run(q, k, v, do, cu, True, v_fold="diagonal")
    first = np.r_[0:128, 300:400]                       # query tile 0 of each document
    assert np.array_equal(fa["O"][first], fd["O"][first]) and np.array_equal(fa["lse"][:, first], fd["lse"][:, first])
    assert not np.array_equal(fa["O"][128:300], fd["O"][128:300])
    Ox, _ = X.forward(q, k, v, cu)
    rel = lambda a, b: np.linalg.norm(a - b) / np.linalg.norm(b)
    assert rel(fd["O"], Ox) < 1.5 * rel(fa["O"], Ox)
    # a future token in the second tile leaves rows of the first tile and the
    # earlier rows of its own tile unchanged
    (f0, b0), (f1, b1) = _future_perturbation(True, ("q", "k", "v", "do"), t=140, L=300, v_fold="diagonal")
    assert np.array_equal(f0["O"][:140], f1["O"][:140]) and np.array_equal(b0["dq"][:140], b1["dq"][:140])
