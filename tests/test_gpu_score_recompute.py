"""The backward recomputes the forward's score tile bit for bit.

FLAMIA Section 3.3 has the backward recompute S and P with the same quantized
representation, tiling, diagonal handling and exponential as the forward.
Here the forward's S and P-hat live only in tensor memory and registers, so
the library's diagnostic hook (flamia_debug_set_score_dump) runs variants of
the attention kernels that copy out one tile: the raw fp32 accumulator of
Qhat Khat^T on the E4M3 codes and the factor 2^(E_Q + E_K) log2(e)/sqrt(d)
each row applies per 32-key group.  The forward's and the backward's copies
must be equal bit for bit; P = 2^(acc * factor - LSE2) then follows from the
same fp32 values and the forward's LSE.

The copies are also checked against the saved codes (the accumulator is their
product up to fp32 accumulation) and the scale bytes (the factor is exactly
fp32(log2(e)/sqrt(d)) 2^(E_Q + E_K)), so the tile is the one asked for.
"""
import math

import numpy as np
import pytest
import torch

import precision_causal_attention_gb300 as F
import workloads as W
from oracle import formats as OF

pytestmark = pytest.mark.gpu

# (query head, document, query tile, key tile): a fully visible tile, the
# partial diagonal tile at a document's end, and a tile of a second document
TILES = [(3, 0, 4, 1), (1, 0, 5, 5), (2, 1, 2, 0)]


def _e4m3_values(codes):
    return np.asarray(OF.e4m3_value(codes), np.float64)


@pytest.mark.parametrize("d", [64, 128])
def test_backward_score_tile_equals_forward_bitwise(d):
    w = W.custom([700, 300, 129], Hq=4, Hkv=2, d=d, seed=50 + d, T=1200)
    dev = torch.device("cuda:0")
    q, k, v, do = (w.tensors[n].to(dev) for n in ("q", "k", "v", "do"))
    cu = torch.from_numpy(np.asarray(w.cu_seqlens, np.int32)).to(dev)
    B = F.Buffers(w.T, w.n_docs, w.Hq, w.Hkv, w.d)
    g = w.Hq // w.Hkv
    try:
        for (h, doc, qt, kt) in TILES:
            bufs = [torch.full(shape, float("nan"), device=dev) for shape in ((128, 128), (128, 4)) * 2]
            F.flamia_debug_set_score_dump(*bufs, h=h, doc=doc, qt=qt, kt=kt)
            F.flamia_fwd(q, k, v, cu, B.out, B.lse, B.saved, B.work)
            F.flamia_bwd(B.out, B.lse, do, cu, B.saved, B.dq, B.dk, B.dv, B.work)
            torch.cuda.synchronize()
            assert F.flamia_get_status() == 0
            s_f, f_f, s_b, f_b = (x.cpu().numpy() for x in bufs)
            assert np.isfinite(s_f).all() and np.isfinite(f_f).all(), "forward copy incomplete"
            assert np.array_equal(s_f.view(np.uint32), s_b.view(np.uint32)), (h, doc, qt, kt)
            assert np.array_equal(f_f.view(np.uint32), f_b.view(np.uint32)), (h, doc, qt, kt)

            # the tile asked for: code products (tokens past T read as zero)
            sv = F.saved_views(B.saved, w.T, w.Hq, w.Hkv, w.d)
            s0 = int(w.cu_seqlens[doc])
            L = int(w.cu_seqlens[doc + 1]) - s0
            rows = s0 + qt * 128 + np.arange(128)
            keys = s0 + kt * 128 + np.arange(128)
            qc = np.zeros((128, d)); kc = np.zeros((128, d))
            okr, okk = rows < w.T, keys < w.T
            qc[okr] = _e4m3_values(sv["q_codes"].cpu().numpy()[rows[okr], h])
            kc[okk] = _e4m3_values(sv["k_codes"].cpu().numpy()[keys[okk], h // g])
            want = qc @ kc.T
            err = np.abs(s_f - want).max() / max(np.abs(want).max(), 1.0)
            assert err < 1e-5, err
            # the factors: exact powers of two times fp32(log2(e) / sqrt(d))
            qs = sv["q_scales"].cpu().numpy()[h]
            ks = sv["k_scales"].cpu().numpy()[h // g]
            base = np.float32(math.log2(math.e) / math.sqrt(d))
            r_in = (qt * 128 + np.arange(128)) < L
            eq = np.where(r_in, qs[np.minimum(rows, w.T - 1)].astype(np.int64) - 127, 0)
            gk = kt * 128 + 32 * np.arange(4)
            ek = np.where(gk < L, ks[np.minimum(s0 + gk, w.T - 1)].astype(np.int64) - 127, 0)
            f_want = (np.float64(base) * np.exp2((eq[:, None] + ek[None, :]).astype(np.float64))).astype(np.float32)
            assert np.array_equal(f_f, f_want), (h, doc, qt, kt)
    finally:
        F.flamia_debug_set_score_dump()
