"""The seeded input recipe: document lengths, packing, shapes and the outlier
construction of the synthetic workloads (FLAMIA Section 4.1, packed documents;
the Llama-1B shape of Section 4.6).  CPU only; small instances of the same
generators where the full ones would only be slower."""
import numpy as np
import torch

import workloads as W


def _rows_end_on_boundaries(w, row_len):
    cu = set(np.asarray(w.cu_seqlens).tolist())
    return all(r * row_len in cu for r in range(w.T // row_len + 1))


def test_tiny_is_the_hand_listed_case():
    w = W.tiny()
    assert list(w.cu_seqlens) == [0, 96, 160, 256]
    assert (w.T, w.Hq, w.Hkv, w.d) == (256, 2, 2, 64)
    assert all(t.dtype == torch.bfloat16 for t in w.tensors.values())


def test_greedy_packing_truncates_only_the_last_document():
    assert W.pack_greedy(iter([300, 500, 400, 100]), 1000) == [300, 500, 200]
    assert W.pack_greedy(iter([1000, 7]), 1000) == [1000]
    assert W.pack_greedy(iter([0, 600, 600]), 1000) == [600, 400]   # empty draws are skipped


def test_packed_llama_shape_lengths_and_rows():
    w = W.llama1b_packed(seed=0, rows=2, row_len=4096)
    assert (w.T, w.Hq, w.Hkv, w.d) == (8192, 32, 8, 64)
    assert _rows_end_on_boundaries(w, 4096)
    L = w.doc_lengths
    assert L.sum() == w.T and L.min() >= 1 and L.max() <= 4096
    # only the last document of a row can fall below the clip floor of 32
    ends = set(np.cumsum(L).tolist())
    short = [i for i, l in enumerate(L) if l < 32]
    assert all(int(np.cumsum(L)[i]) % 4096 == 0 for i in short) and 4096 in ends
    for n, shp in (("q", (8192, 32, 64)), ("k", (8192, 8, 64)), ("v", (8192, 8, 64)), ("do", (8192, 32, 64))):
        assert tuple(w.tensors[n].shape) == shp


def test_lognormal_median_is_about_1024():
    rng = np.random.default_rng(0)
    g = W._lognormal_lengths(rng, 1024, 1.0, 32, 8192)
    draws = np.array([next(g) for _ in range(20000)])
    assert 950 < np.median(draws) < 1100
    assert draws.min() >= 32 and draws.max() <= 8192


def test_seeds_are_deterministic_and_distinct():
    a = W.llama1b_packed(seed=3, rows=1, row_len=2048)
    b = W.llama1b_packed(seed=3, rows=1, row_len=2048)
    c = W.llama1b_packed(seed=4, rows=1, row_len=2048)
    assert np.array_equal(a.cu_seqlens, b.cu_seqlens) and torch.equal(a.tensors["q"], b.tensors["q"])
    assert not np.array_equal(a.cu_seqlens, c.cu_seqlens)


def test_batched_is_one_document_per_row():
    w = W.llama1b_batched(seed=0, rows=3, row_len=1024)
    assert list(w.cu_seqlens) == [0, 1024, 2048, 3072]


def test_skewed_rows_end_with_the_long_document():
    w = W.skewed(seed=0, rows=2, row_len=4096, long_len=2048)
    cu = np.asarray(w.cu_seqlens)
    L = w.doc_lengths
    assert _rows_end_on_boundaries(w, 4096)
    for r in range(2):
        # the document ending at the row end is the long one, starting half-way
        i = int(np.where(cu == (r + 1) * 4096)[0][0]) - 1
        assert L[i] == 2048 and cu[i] == r * 4096 + 2048
    short = [l for l in L if l != 2048]
    assert max(short) <= 512
    assert sum(l < 64 for l in short) <= 2                   # only a row's truncated last short document


def test_outlier_channels_and_tokens():
    w = W.outliers(seed=0, rows=1, row_len=4096)
    q = w.tensors["q"].float()
    v = w.tensors["v"].float()
    # per-channel median magnitude (the 0.1 % outlier tokens do not move it):
    # four channels per head stand out by about x20; V is untouched
    ch = q.abs().median(dim=0).values                          # [H, d]
    top = torch.topk(ch, 4, dim=1).values
    rest = torch.sort(ch, dim=1).values[:, :-4]
    assert torch.all(top.min(dim=1).values > 10.0 * rest.max(dim=1).values)
    vm = v.abs().median(dim=0).values
    assert vm.max() < 1.5 * vm.min()
    # 0.1 % of the tokens are scaled by 50 in every head
    tok_norm = q.norm(dim=(1, 2))
    n_out = int(round(0.001 * w.T))
    big = torch.topk(tok_norm, n_out + 1).values
    assert big[n_out - 1] > 10.0 * torch.median(tok_norm) and big[n_out] < 5.0 * torch.median(tok_norm)
