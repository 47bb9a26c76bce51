"""Document-local token-block quantization of packed [T, H, d] tensors.

Source: "FLAMIA: FLAsh MIcroscaling Attention ..." Section 3.1 (token-block
scaling: one power-of-two exponent shared by 32 consecutive tokens and the
full head dimension, per head), Section 3.2 (round the exponent up, so no
element is clamped), Section 3.6.1 (quantizers work on the packed layout,
keep token blocks inside document boundaries and write one scale entry per
token).

Reading taken where the pages leave it open: block b of document [s, e)
covers tokens [s + 32 b, min(s + 32 b + 32, e)) (document-relative blocks; the
last block of a document may be short).  Tokens outside every document are
not quantized.

Exact options (Appendix A.3): per-token operand scales give every token of
every head its own exponent, sized from that token's d elements only.

Pinned by tests/test_oracle_blocks.py: brute-force per-block search of the
smallest admissible exponent, the 2^k shift invariance, block boundaries
against hand-listed cases, and independence of documents; the per-token form
against the block form with every token its own one-token document.
"""
from __future__ import annotations

import numpy as np

from .formats import e4m3_encode, e4m3_value, roundup_exponent, floor_exponent, scale_byte, SCALE_EXP_MIN

BLOCK = 32


def doc_blocks(cu_seqlens):
    """Yield (doc, first_token, end_token) for every 32-token block, document-relative."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    for r in range(len(cu) - 1):
        s, e = int(cu[r]), int(cu[r + 1])
        for b0 in range(s, e, BLOCK):
            yield r, b0, min(b0 + BLOCK, e)


def quantize_token_blocks(x, cu_seqlens, rule: str = "roundup"):
    """Quantize x [T, H, d] (exact values as float64) with document-local token blocks.

    Returns (codes uint8 [T, H, d], scale bytes uint8 [H, T], exponents int64 [H, T]).
    Tokens outside every document keep code 0 and exponent -127 (scale byte 0);
    they are never read.
    """
    x = np.asarray(x, dtype=np.float64)
    T, H, d = x.shape
    expo_fn = roundup_exponent if rule == "roundup" else floor_exponent
    codes = np.zeros((T, H, d), dtype=np.uint8)
    E_tok = np.full((H, T), SCALE_EXP_MIN, dtype=np.int64)
    for _, b0, b1 in doc_blocks(cu_seqlens):
        blk = x[b0:b1]                                   # [n, H, d]
        amax = np.abs(blk).max(axis=(0, 2))              # [H]
        E = expo_fn(amax)                                # [H]
        codes[b0:b1] = e4m3_encode(np.ldexp(blk, -E[None, :, None]))
        E_tok[:, b0:b1] = E[:, None]
    return codes, scale_byte(E_tok), E_tok


def quantize_per_token(x, cu_seqlens, rule: str = "roundup"):
    """Quantize x [T, H, d] with one exponent per (token, head): the per-token
    operand scales of the exact options.  Same outputs and conventions as
    quantize_token_blocks."""
    x = np.asarray(x, dtype=np.float64)
    T, H, d = x.shape
    expo_fn = roundup_exponent if rule == "roundup" else floor_exponent
    codes = np.zeros((T, H, d), dtype=np.uint8)
    E_tok = np.full((H, T), SCALE_EXP_MIN, dtype=np.int64)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    for r in range(len(cu) - 1):
        s, e = int(cu[r]), int(cu[r + 1])
        if e <= s:
            continue
        blk = x[s:e]                                     # [n, H, d]
        E = expo_fn(np.abs(blk).max(axis=2))             # [n, H]
        codes[s:e] = e4m3_encode(np.ldexp(blk, -E[:, :, None]))
        E_tok[:, s:e] = E.T
    return codes, scale_byte(E_tok), E_tok


def dequantize(codes, E_tok):
    """Values represented by token-block codes: val(code) * 2^E (layouts as above)."""
    v = e4m3_value(codes)                                # [T, H, d]
    return np.ldexp(v, np.asarray(E_tok).T[:, :, None])


def in_doc_mask(cu_seqlens, T: int) -> np.ndarray:
    """Boolean [T]: token lies inside some document."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    m = np.zeros(T, dtype=bool)
    m[int(cu[0]):int(cu[-1])] = True
    return m
