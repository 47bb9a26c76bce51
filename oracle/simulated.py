"""Quantization-simulating attention: the MXFP8 path computed exactly in fp64.

Source: "FLAMIA: FLAsh MIcroscaling Attention ..." (arXiv 2611.03344).

Forward, per document, query head and 128-query tile (Sections 3.4, 3.5.1, 3.6,
Appendix B.1):
  1. Q, K, V are quantized with document-local token blocks (oracle.blocks).
  2. S2_ij = (sum_k qhat_ik khat_jk) * log2(e) / sqrt(d) for visible keys
     (same document; j <= i when causal).  The code dot product is exact in
     fp64: E4M3 products have at most 8 significant bits and the partial sums
     of d <= 128 of them stay far inside 53 bits.
  3. Key tiles of 128 document-relative keys are visited in a fixed order:
     causal calls take the fully visible tiles from qt-1 down to 0 and the
     diagonal tile qt last; non-causal calls go from the last tile down to 0.
     Per query row: m = -inf, l = 0, acc = 0.  For each tile, with t the row
     maximum of the visible S2 in it: if m = -inf or t - m > tau, rescale acc
     and l by 2^(m - t) and set m = t (conditional rescaling, decided per row).
     Then p~ = 2^(S2 - m), l += sum p~, Phat = E4M3(2^c p~) 2^-c and
     acc += Phat Vhat.
  4. O = acc / l, LSE = (m + log2 l) ln 2.  Rows outside every document keep
     O = 0 and LSE = +inf (Section 3.6.1).
  Variant ``exact_max``: m is the true row maximum from the start (one pass).

Backward (Sections 2, 3.3, Appendix B.1):
  D_i = sum_k dOhat_ik O_ik with the forward's bf16 output O and the
  token-block-quantized dO; P = 2^(S2 - LSE log2 e) from the same S2;
  dP = dOhat Vhat^T; dS = P o (dP - D) (zero where masked); dS is quantized
  per 32 x 32 document-relative (query block, key block) with the round-up
  exponent; P' = E4M3(2^8 P) 2^-8; dV_j = sum_i P'_ij dOhat_i,
  dK_j = sum_i dShat_ij Qhat_i / sqrt(d), dQ_i = sum_j dShat_ij Khat_j / sqrt(d);
  dK and dV also sum over the query heads of a grouped-query group.

Readings where the pages are silent (each is listed with the design notes):
  * tau is in log2 units and the rescale decision is made per query row;
  * the row sum l accumulates the unquantized p~ (quantized probabilities
    need not sum to one, Section 3.3);
  * LSE is in natural-log units, layout [Hq, T];
  * P for the backward is 2^(S2 - LSE2) with the forward's LSE (Section 3.3:
    same representations, exponential and row-maximum convention).

Option ``hadamard`` (Section 3.4, Appendix A.2; oracle.hadamard): Q and K are
rotated along the head dimension by the Sylvester matrix H_d before their
quantization, the scores take the factor 1/d out, and dQ, dK are computed for
the rotated operands and mapped back with H_d / d.

Option ``exact`` (the exact options, Section 3.2 and Appendices A.1 and A.3):
every scale of an operand is sized from data that every row reading it may see,
so a later token of the same document changes no bit of an earlier row's O,
LSE or dQ.
  * Q, K, V and dO get per-token exponents (oracle.blocks.quantize_per_token).
  * Forward: V's per-key exponent is folded into P-hat.  For query row i and
    the 32-key group g of a tile, G_ig is the largest V exponent among the
    keys of g that row i sees, sigma_ig = max(G_ig - c, -127) is the P-hat
    block scale, and the code is E4M3(p~_ij 2^(E_V(j) - sigma_ig)) (at most
    2^(c + tau), as in the default path); it multiplies 2^sigma_ig times
    V's code.
  * Backward, dQ (the K fold and the per-query-row dS exponent):
    x_ij = dS_ij 2^E_K(j) is quantized with one exponent per (query row,
    32-key group) and multiplies K's codes.
  * Backward, dK and dV.  dK_j and dV_j depend on later queries by
    definition, so their payloads have no causal constraint and keep
    block-shaped scales over in-document values, with the per-token exponent
    of the contracted operand folded in.  dK uses y_ij = dS_ij 2^E_Q(i) in
    32 x 32 blocks.  dV uses E4M3(2^8 P_ij 2^(E_dO(i) - H_b)), where H_b is
    the largest dO exponent of the 32-query block.
  fp32 dQ accumulation has no prescale, so the pages' causal dQ scale (A.4)
  has nothing to act on here.
  ``v_fold="diagonal"`` restricts the V fold to the diagonal tile of a
  causal call, as the pages do (Section 3.2).  The other tiles hold only
  keys before every query of the tile, so they keep V's token-block codes
  and the fixed 2^c multiplier; so does dP.  A non-causal call has no
  diagonal, and every tile then uses the block codes.

Option ``scores="nvfp4"`` (the mixed NVFP4/FP8 path, Sections 3.4 and 3.5.2;
oracle.nvfp4): S and its recomputation use NVFP4 Q and K (E2M1 codes, one
UE4M3 scale per 16 head-dimension elements of each token).  dQ and dK still
use the E4M3 token-block Q and K.  P-hat is quantized in the log domain: for
query row i and 32-key group g, let xmax be the largest exponent argument
S2 - m among the keys the row sees.  Then E_ig = roundup(2^xmax) (the
round-up rule of Section 3.2 applied to the group's largest probability,
using max_j 2^x_j = 2^(max_j x_j)), and the code is E4M3(2^(x - E_ig)),
scaled by 2^E_ig.  The fixed multiplier 2^c is not used on this path.

Switches ``quantize`` / ``p_quant`` / ``ds_quant`` replace each quantizer by the
identity; with all off and ``exact_max`` the result equals oracle.exact up to
fp64 rounding (tests/test_oracle_simulated.py).  The fp32 intermediates of a
GPU (exp, S2, dS) make its P-hat and dS-hat codes differ near rounding ties:
those codes are *parity unpinned* and compared by tolerance only.
"""
from __future__ import annotations

import math

import numpy as np

from .blocks import quantize_token_blocks, quantize_per_token, dequantize
from . import hadamard as HD
from . import nvfp4 as NV
from .formats import quantize_value, roundup_exponent, floor_exponent, e4m3_encode, e4m3_value, bf16_round

LOG2E = 1.0 / math.log(2.0)
LN2 = math.log(2.0)
TILE = 128
DS_BLOCK = 32


def _doc_ranges(cu_seqlens):
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    return [(int(cu[r]), int(cu[r + 1])) for r in range(len(cu) - 1)]


def quantize_inputs(x, cu_seqlens, quantize: bool = True, rule: str = "roundup", per_token: bool = False):
    """(dequantized values, codes, scale bytes [H, T], exponents [H, T]) of a [T, H, d] tensor.

    Without quantization the exponents are all 0 (so the exact options' folds
    multiply by 1)."""
    x = np.asarray(x, dtype=np.float64)
    if not quantize:
        return x, None, None, np.zeros((x.shape[1], x.shape[0]), np.int64)
    quant = quantize_per_token if per_token else quantize_token_blocks
    codes, sbytes, E = quant(x, cu_seqlens, rule=rule)
    return dequantize(codes, E), codes, sbytes, E


def key_tile_order(qt: int, nt: int, causal: bool):
    """Key tiles a query tile visits, in visiting order.

    Causal: the fully visible tiles qt-1 .. 0, then the diagonal tile qt (so the
    first tile a row sees holds 128 keys and the running maximum starts close to
    the final one).  Non-causal: nt-1 down to 0.
    """
    if causal:
        return list(range(qt - 1, -1, -1)) + [qt]
    return list(range(nt - 1, -1, -1))


def forward(q, k, v, cu_seqlens, causal: bool = True, c: int = 4, tau: float = 4.0, heads=None,
            quantize: bool = True, p_quant: bool = True, exact_max: bool = False, rule: str = "roundup",
            q_tiles=None, prequantized=None, hadamard: bool = False, exact: bool = False,
            scores: str = "mxfp8", v_fold: str = "all"):
    """Simulated MXFP8 (or mixed NVFP4/FP8) forward.

    Returns a dict with O (float64, unrounded), O_bf16, lse [Hq, T], the quantized
    inputs (codes / scale bytes / exponents of q, k, v) and ``pmax``, the largest
    2^c p~ fed to the probability quantizer (the saturation check of Appendix B.1).
    ``q_tiles``: optional set of (doc, qtile) pairs to compute (others stay NaN).
    """
    q = np.asarray(q, np.float64)
    T, Hq, d = q.shape
    Hkv = np.asarray(k).shape[1]
    g = Hq // Hkv
    if prequantized is None:
        qr = HD.rotate(q) if hadamard else q
        kr = HD.rotate(k) if hadamard else k
        qh, qc, qs, qE = quantize_inputs(qr, cu_seqlens, quantize, rule, exact)
        kh, kc, ks, kE = quantize_inputs(kr, cu_seqlens, quantize, rule, exact)
        vh, vc, vs, vE = quantize_inputs(v, cu_seqlens, quantize, rule, exact)
    else:
        (qh, qc, qs, qE), (kh, kc, ks, kE), (vh, vc, vs, vE) = prequantized
    assert scores in ("mxfp8", "nvfp4") and not (scores == "nvfp4" and exact)
    assert v_fold in ("all", "diagonal")
    vhb = quantize_inputs(v, cu_seqlens, quantize, rule)[0] if exact and v_fold == "diagonal" else None
    q4 = k4 = None
    qsc, ksc = qh, kh                                  # the operands of the score products
    if scores == "nvfp4" and quantize:
        q4 = NV.quantize_nvfp4(HD.rotate(q) if hadamard else q, cu_seqlens)
        k4 = NV.quantize_nvfp4(HD.rotate(k) if hadamard else k, cu_seqlens)
        qsc, ksc = q4[2], k4[2]
    heads = range(Hq) if heads is None else heads
    O = np.zeros((T, Hq, d))
    lse = np.full((Hq, T), np.inf)
    scale = LOG2E / math.sqrt(d) / (d if hadamard else 1)
    pmax = 0.0
    gmin = np.inf                      # smallest largest-P-hat-input of a (row, 32-key group) that sees a key
    two_c = 2.0 ** c
    for r, (s, e) in enumerate(_doc_ranges(cu_seqlens)):
        L = e - s
        if L <= 0:
            continue
        nt = (L + TILE - 1) // TILE
        for qt in range(nt):
            if q_tiles is not None and (r, qt) not in q_tiles:
                O[s + qt * TILE:s + min(qt * TILE + TILE, L)] = np.nan
                continue
            i0, i1 = qt * TILE, min(qt * TILE + TILE, L)
            ii = np.arange(i0, i1)
            for h in heads:
                hk = h // g
                Q = qsc[s + i0:s + i1, h]
                n = i1 - i0
                m = np.full(n, -np.inf)
                l = np.zeros(n)
                acc = np.zeros((n, d))
                order = key_tile_order(qt, nt, causal)
                if exact_max:
                    kend = i1 if causal else L
                    S_all = (Q @ ksc[s:s + kend, hk].T) * scale
                    if causal:
                        S_all = np.where(np.arange(kend)[None, :] <= ii[:, None], S_all, -np.inf)
                    m = S_all.max(axis=1)
                for kt in order:
                    j0, j1 = kt * TILE, min(kt * TILE + TILE, L)
                    K = ksc[s + j0:s + j1, hk]
                    # the V fold on this tile (exact options): every tile, or
                    # only the diagonal one with block-coded V elsewhere
                    fold_v = exact and (v_fold == "all" or (causal and kt == qt))
                    V = (vh if fold_v or vhb is None else vhb)[s + j0:s + j1, hk]
                    S2 = (Q @ K.T) * scale
                    if causal:
                        S2 = np.where(np.arange(j0, j1)[None, :] <= ii[:, None], S2, -np.inf)
                    if not exact_max:
                        t = S2.max(axis=1)
                        upd = np.isneginf(m) | (t - m > tau)
                        m_new = np.where(upd, t, m)
                        alpha = np.where(np.isneginf(m), 0.0, np.exp2(np.where(upd, m - m_new, 0.0)))
                        acc *= alpha[:, None]
                        l *= alpha
                        m = m_new
                    pt = np.exp2(S2 - m[:, None])
                    l += pt.sum(axis=1)
                    if scores == "nvfp4":
                        # log-domain P-hat: per (row, 32-key group) the
                        # exponent of the group's largest probability
                        xarg = S2 - m[:, None]
                        grp = np.arange(j1 - j0) // DS_BLOCK
                        fold = np.zeros(S2.shape)
                        for gq in range(grp[-1] + 1):
                            cols = grp == gq
                            xmax = xarg[:, cols].max(axis=1)
                            Eg = roundup_exponent(np.exp2(xmax))
                            fold[:, cols] = np.ldexp(1.0, -Eg)[:, None]
                        scaled = pt * fold
                    elif fold_v:
                        # per (row, 32-key group): P-hat scale from the V
                        # exponents of the keys the row sees
                        ev = vE[hk, s + j0:s + j1]
                        vis = np.ones(S2.shape, bool)
                        if causal:
                            vis = np.arange(j0, j1)[None, :] <= ii[:, None]
                        grp = np.arange(j1 - j0) // DS_BLOCK
                        sigma = np.zeros(S2.shape, np.int64)
                        for gq in range(grp[-1] + 1):
                            cols = grp == gq
                            G = np.where(vis[:, cols], ev[cols][None, :], -(1 << 30)).max(axis=1)
                            sigma[:, cols] = np.maximum(G - c, -127)[:, None]
                        fold = np.ldexp(1.0, ev[None, :] - sigma)
                        scaled = pt * fold
                    else:
                        fold = two_c
                        scaled = two_c * pt
                    pmax = max(pmax, float(scaled.max()))
                    for gq in range(0, j1 - j0, DS_BLOCK):
                        blk = scaled[:, gq:gq + DS_BLOCK]
                        seen = np.isfinite(S2[:, gq:gq + DS_BLOCK]).any(axis=1)
                        if seen.any():
                            gmin = min(gmin, float(blk[seen].max(axis=1).min()))
                    if p_quant:
                        Ph = quantize_value(scaled) / fold
                    else:
                        Ph = pt
                    acc += Ph @ V
                O[s + i0:s + i1, h] = acc / l[:, None]
                lse[h, s + i0:s + i1] = (m + np.log2(l)) * LN2
    return {
        "O": O, "O_bf16": bf16_round(O), "lse": lse, "pmax": pmax, "p_group_max_min": gmin,
        "q": (qh, qc, qs, qE), "k": (kh, kc, ks, kE), "v": (vh, vc, vs, vE),
        "q_nvfp4": q4, "k_nvfp4": k4,
    }


def ds_quantize(dS, rule: str = "roundup"):
    """32 x 32 block quantization of dS [n, m] whose rows and columns start on block boundaries.

    Returns (values, codes, exponents [ceil(n/32), ceil(m/32)]).
    """
    n, m = dS.shape
    nb, mb = -(-n // DS_BLOCK), -(-m // DS_BLOCK)
    pad = np.zeros((nb * DS_BLOCK, mb * DS_BLOCK))
    pad[:n, :m] = dS
    blk = pad.reshape(nb, DS_BLOCK, mb, DS_BLOCK)
    amax = np.abs(blk).max(axis=(1, 3))
    E = (roundup_exponent if rule == "roundup" else floor_exponent)(amax)
    scaled = np.ldexp(blk, -E[:, None, :, None])
    codes = e4m3_encode(scaled)
    vals = np.ldexp(e4m3_value(codes), E[:, None, :, None])
    return vals.reshape(nb * DS_BLOCK, mb * DS_BLOCK)[:n, :m], codes.reshape(nb * DS_BLOCK, mb * DS_BLOCK)[:n, :m], E


def ds_quantize_rows(x, rule: str = "roundup"):
    """Quantization of x [n, m] with one exponent per (row, 32-column group),
    the groups starting at column 0: the per-query-row dS exponent of the
    exact options.  Returns (values, codes, exponents [n, ceil(m/32)])."""
    n, m = x.shape
    mb = -(-m // DS_BLOCK)
    pad = np.zeros((n, mb * DS_BLOCK))
    pad[:, :m] = x
    blk = pad.reshape(n, mb, DS_BLOCK)
    E = (roundup_exponent if rule == "roundup" else floor_exponent)(np.abs(blk).max(axis=2))
    codes = e4m3_encode(np.ldexp(blk, -E[:, :, None]))
    vals = np.ldexp(e4m3_value(codes), E[:, :, None])
    return vals.reshape(n, mb * DS_BLOCK)[:, :m], codes.reshape(n, mb * DS_BLOCK)[:, :m], E


def quantize_do(do, O_bf16, cu_seqlens, quantize: bool = True, rule: str = "roundup", per_token: bool = False):
    """Quantized dO (token blocks, or per token) and D_i = sum_k dOhat_ik O_ik
    (D layout [Hq, T], 0 outside documents)."""
    doh, doc_, dos, doE = quantize_inputs(do, cu_seqlens, quantize, rule, per_token)
    O = np.asarray(O_bf16, np.float64)
    D = np.einsum("thd,thd->ht", doh, np.nan_to_num(O))
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    D[:, :int(cu[0])] = 0.0
    D[:, int(cu[-1]):] = 0.0
    return (doh, doc_, dos, doE), D


def backward(q, k, v, O_bf16, lse, do, cu_seqlens, causal: bool = True, heads=None, quantize: bool = True,
             p_quant: bool = True, ds_quant: bool = True, p_bwd_exp: int = 8, rule: str = "roundup",
             prequantized=None, hadamard: bool = False, exact: bool = False, scores: str = "mxfp8",
             v_fold: str = "all"):
    """Simulated MXFP8 (or mixed NVFP4/FP8) backward.  Returns dict with dq, dk, dv (float64), their bf16 roundings, D, dO codes.

    ``prequantized``: (Q, K, V) values, or with ``exact`` the (values,
    exponents [H, T]) pairs of the three."""
    q = np.asarray(q, np.float64)
    T, Hq, d = q.shape
    Hkv = np.asarray(k).shape[1]
    g = Hq // Hkv
    if prequantized is None:
        qh, _, _, qE = quantize_inputs(HD.rotate(q) if hadamard else q, cu_seqlens, quantize, rule, exact)
        kh, _, _, kE = quantize_inputs(HD.rotate(k) if hadamard else k, cu_seqlens, quantize, rule, exact)
        vh = quantize_inputs(v, cu_seqlens, quantize, rule, exact)[0]
    elif exact:
        (qh, qE), (kh, kE), (vh, _) = prequantized
    else:
        qh, kh, vh = prequantized
    do_pack, D = quantize_do(do, O_bf16, cu_seqlens, quantize, rule, exact)
    doh, doE = do_pack[0], do_pack[3]
    assert scores in ("mxfp8", "nvfp4") and not (scores == "nvfp4" and exact)
    assert v_fold in ("all", "diagonal")
    vhb = quantize_inputs(v, cu_seqlens, quantize, rule)[0] if exact and v_fold == "diagonal" else None
    qsc, ksc = qh, kh                                  # score recomputation operands
    if scores == "nvfp4" and quantize:
        qsc = NV.quantize_nvfp4(HD.rotate(q) if hadamard else q, cu_seqlens)[2]
        ksc = NV.quantize_nvfp4(HD.rotate(k) if hadamard else k, cu_seqlens)[2]
    heads = range(Hq) if heads is None else heads
    dq = np.zeros((T, Hq, d)); dk = np.zeros((T, Hkv, d)); dv = np.zeros((T, Hkv, d))
    scale = LOG2E / math.sqrt(d) / (d if hadamard else 1)
    pe = 2.0 ** p_bwd_exp
    for s, e in _doc_ranges(cu_seqlens):
        L = e - s
        if L <= 0:
            continue
        for h in heads:
            hk = h // g
            K = kh[s:e, hk]; V = vh[s:e, hk]
            for i0 in range(0, L, TILE):
                i1 = min(i0 + TILE, L)
                ii = np.arange(i0, i1)
                kend = i1 if causal else L
                Q = qh[s + i0:s + i1, h]
                dO = doh[s + i0:s + i1, h]
                S2 = (qsc[s + i0:s + i1, h] @ ksc[s:s + kend, hk].T) * scale
                lse2 = lse[h, s + i0:s + i1] * LOG2E
                with np.errstate(over="ignore"):     # masked entries may overflow before masking
                    P = np.exp2(S2 - lse2[:, None])
                if causal:
                    P = np.where(np.arange(kend)[None, :] <= ii[:, None], P, 0.0)
                if vhb is None:
                    Vp = V[:kend]
                else:
                    # block-coded V before the diagonal tile (per-token V on it
                    # for a causal call; block codes everywhere otherwise)
                    d0 = i0 if causal else kend
                    Vp = np.concatenate([vhb[s:s + d0, hk], V[d0:kend]])
                dP = dO @ Vp.T
                dS = P * (dP - D[h, s + i0:s + i1][:, None])
                if not ds_quant:
                    dShQ = dShK = dS
                elif exact:
                    # dQ payload: K fold, one exponent per (query row, 32-key group)
                    fk = np.ldexp(1.0, kE[hk, s:s + kend])[None, :]
                    dShQ = ds_quantize_rows(dS * fk, rule)[0] / fk
                    # dK payload: Q fold, 32 x 32 blocks
                    fq = np.ldexp(1.0, qE[h, s + i0:s + i1])[:, None]
                    dShK = ds_quantize(dS * fq, rule)[0] / fq
                else:
                    dShQ = dShK = ds_quantize(dS, rule)[0]
                if not p_quant:
                    Pq = P
                elif exact:
                    # dV payload: dO fold, scale per 32-query block
                    eo = doE[h, s + i0:s + i1]
                    Hb = np.array([eo[b:b + DS_BLOCK].max() for b in range(0, i1 - i0, DS_BLOCK)])
                    sig = np.maximum(np.repeat(Hb, DS_BLOCK)[:i1 - i0] - p_bwd_exp, -127)
                    fo = np.ldexp(1.0, eo - sig)[:, None]
                    Pq = quantize_value(P * fo) / fo
                else:
                    Pq = quantize_value(pe * P) / pe
                dq[s + i0:s + i1, h] = dShQ @ K[:kend] / math.sqrt(d)
                dk[s:s + kend, hk] += dShK.T @ Q / math.sqrt(d)
                dv[s:s + kend, hk] += Pq.T @ dO
    if hadamard:
        # gradients of the rotated operands, mapped back
        dq = HD.unrotate(dq)
        dk = HD.unrotate(dk)
    return {"dq": dq, "dk": dk, "dv": dv, "dq_bf16": bf16_round(dq), "dk_bf16": bf16_round(dk),
            "dv_bf16": bf16_round(dv), "D": D, "do": do_pack}
