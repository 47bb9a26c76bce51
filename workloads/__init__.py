"""Seeded synthetic inputs for packed causal attention.

This module holds no attention or quantization arithmetic: it only draws
document lengths, packs them into rows and draws Q, K, V, dO.  Both the CPU
oracle (``oracle/``) and the CUDA path consume these inputs, so the two never
share any code beyond this generator.

Recipe (identical for every workload):

* Document lengths come from ``numpy.random.default_rng(seed)``.  A row of
  ``row_len`` tokens is filled greedily: draw a length, append
  ``min(draw, remaining)``, repeat until the row is full (so the last document
  of a row may be truncated).  Rows are concatenated into one packed sequence
  of ``T = rows * row_len`` tokens; ``cu_seqlens`` has the document starts.
* Tensors come from ``torch.Generator().manual_seed(seed)``: ``randn`` in fp32,
  cast to bf16, drawn in the order q, k, v, dO with shapes [T, H, d]
  (the packed "varlen" layout).
* The outlier workload then scales, in Q and K, four fixed channels per head
  (drawn from the numpy generator) by 20 and 0.1 % of the tokens (all heads)
  by 50, before the bf16 cast.

The five named workloads follow the shapes of the packed-document experiments
in "FLAMIA: FLAsh MIcroscaling Attention ..." (Section 4.1, packed documents;
Llama-style 1B pretraining shape of Section 4.6).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np
import torch


@dataclass
class Workload:
    name: str
    cu_seqlens: np.ndarray          # int32 [n_docs + 1]
    T: int                          # packed tokens (buffer rows)
    Hq: int
    Hkv: int
    d: int
    causal: bool = True
    tensors: Dict[str, torch.Tensor] = field(default_factory=dict)  # q, k, v, do (bf16, CPU)
    description: str = ""

    @property
    def n_docs(self) -> int:
        return int(len(self.cu_seqlens) - 1)

    @property
    def doc_lengths(self) -> np.ndarray:
        return np.diff(self.cu_seqlens).astype(np.int64)


def pack_greedy(draws, row_len: int) -> List[int]:
    """Fill one row of ``row_len`` tokens with lengths taken from ``draws``."""
    out: List[int] = []
    remaining = row_len
    for x in draws:
        if remaining <= 0:
            break
        take = int(min(int(x), remaining))
        if take <= 0:
            continue
        out.append(take)
        remaining -= take
    assert remaining == 0, "draw iterator exhausted before the row was full"
    return out


def _lognormal_lengths(rng: np.random.Generator, median: float, sigma: float, lo: int, hi: int):
    while True:
        x = rng.lognormal(mean=np.log(median), sigma=sigma)
        yield int(np.clip(np.round(x), lo, hi))


def _uniform_lengths(rng: np.random.Generator, lo: int, hi: int):
    while True:
        yield int(rng.integers(lo, hi + 1))


def cu_from_lengths(lengths) -> np.ndarray:
    cu = np.zeros(len(lengths) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(lengths)
    return cu.astype(np.int32)


def draw_tensors(T: int, Hq: int, Hkv: int, d: int, seed: int, names=("q", "k", "v", "do")) -> Dict[str, torch.Tensor]:
    g = torch.Generator().manual_seed(seed)
    shapes = {"q": (T, Hq, d), "k": (T, Hkv, d), "v": (T, Hkv, d), "do": (T, Hq, d)}
    out = {}
    for n in ("q", "k", "v", "do"):
        t = torch.randn(shapes[n], generator=g, dtype=torch.float32)
        if n in names:
            out[n] = t
    return out


def _finish(w: Workload, raw: Dict[str, torch.Tensor]) -> Workload:
    w.tensors = {k: v.to(torch.bfloat16).contiguous() for k, v in raw.items()}
    return w


def tiny(seed: int = 0) -> Workload:
    """T=256, documents [96, 64, 96], 2 heads, d=64, MHA."""
    cu = np.array([0, 96, 160, 256], dtype=np.int32)
    w = Workload("tiny_T256_docs96-64-96_h2_d64", cu, 256, 2, 2, 64,
                 description="1 row of 256 tokens, docs [96,64,96], 2 heads MHA, d=64")
    return _finish(w, draw_tensors(256, 2, 2, 64, seed))


def llama1b_packed(seed: int = 0, rows: int = 4, row_len: int = 8192) -> Workload:
    """4 rows x 8192, lognormal(median 1024, sigma 1) lengths clipped to [32, 8192]; 32/8 heads, d=64."""
    rng = np.random.default_rng(seed)
    lens: List[int] = []
    for _ in range(rows):
        lens += pack_greedy(_lognormal_lengths(rng, 1024, 1.0, 32, row_len), row_len)
    T = rows * row_len
    w = Workload(f"llama1b_packed_{rows}x{row_len}_h32kv8_d64", cu_from_lengths(lens), T, 32, 8, 64,
                 description=f"{rows} rows x {row_len}, lognormal(1024,1) docs in [32,{row_len}], Hq=32 Hkv=8 d=64 causal")
    return _finish(w, draw_tensors(T, 32, 8, 64, seed))


def llama1b_batched(seed: int = 0, rows: int = 4, row_len: int = 8192) -> Workload:
    """The Llama-1B shape without packing: 4 sequences of exactly 8192 tokens (a
    fixed-length batch, one document per row); 32/8 heads, d=64."""
    T = rows * row_len
    w = Workload(f"llama1b_batched_{rows}x{row_len}_h32kv8_d64", cu_from_lengths([row_len] * rows), T, 32, 8, 64,
                 description=f"{rows} sequences x {row_len} (one document each), Hq=32 Hkv=8 d=64")
    return _finish(w, draw_tensors(T, 32, 8, 64, seed))


def long_single(seed: int = 0, T: int = 16384) -> Workload:
    """One 16384-token document, 16 MHA heads, d=128."""
    w = Workload(f"long_single_{T}_h16_d128", cu_from_lengths([T]), T, 16, 16, 128,
                 description=f"1 document of {T} tokens, 16 MHA heads, d=128 causal")
    return _finish(w, draw_tensors(T, 16, 16, 128, seed))


def skewed(seed: int = 0, rows: int = 2, row_len: int = 32768, long_len: int = 16384) -> Workload:
    """Each row: uniform[64,512] documents filling row_len-long_len tokens, then one long document."""
    rng = np.random.default_rng(seed)
    lens: List[int] = []
    for _ in range(rows):
        lens += pack_greedy(_uniform_lengths(rng, 64, 512), row_len - long_len)
        lens.append(long_len)
    T = rows * row_len
    w = Workload(f"skewed_{rows}x{row_len}_h16kv4_d128", cu_from_lengths(lens), T, 16, 4, 128,
                 description=f"{rows} rows x {row_len}: uniform[64,512] docs then one {long_len} doc; Hq=16 Hkv=4 d=128")
    return _finish(w, draw_tensors(T, 16, 4, 128, seed))


def outliers(seed: int = 0, rows: int = 2, row_len: int = 16384) -> Workload:
    """lognormal(median 2048) docs in [32, row_len]; Q,K with 4 outlier channels/head (x20) and 0.1 % tokens x50."""
    rng = np.random.default_rng(seed)
    lens: List[int] = []
    for _ in range(rows):
        lens += pack_greedy(_lognormal_lengths(rng, 2048, 1.0, 32, row_len), row_len)
    T = rows * row_len
    H, d = 16, 128
    raw = draw_tensors(T, H, H, d, seed)
    chans = np.stack([rng.choice(d, size=4, replace=False) for _ in range(H)])  # [H, 4]
    n_tok = max(1, int(round(0.001 * T)))
    toks = rng.choice(T, size=n_tok, replace=False)
    for name in ("q", "k"):
        t = raw[name]
        for h in range(H):
            t[:, h, torch.from_numpy(chans[h])] *= 20.0
        t[torch.from_numpy(toks)] *= 50.0
    w = Workload(f"outliers_{rows}x{row_len}_h16_d128", cu_from_lengths(lens), T, H, H, d,
                 description=f"{rows} rows x {row_len}, lognormal(2048,1) docs; Q,K outlier channels x20, 0.1% tokens x50")
    return _finish(w, raw)


def custom(lengths, Hq: int, Hkv: int, d: int, seed: int = 0, T: Optional[int] = None, causal: bool = True,
           name: str = "custom") -> Workload:
    """Arbitrary document lengths (zero-length documents allowed); T >= sum(lengths) adds padding rows."""
    cu = cu_from_lengths(list(lengths))
    total = int(cu[-1])
    T = total if T is None else int(T)
    assert T >= total
    w = Workload(name, cu, T, Hq, Hkv, d, causal=causal, description=f"custom lengths={list(lengths)[:8]}...")
    return _finish(w, draw_tensors(T, Hq, Hkv, d, seed))


NAMED = {
    "tiny": tiny,
    "llama1b_packed": llama1b_packed,
    "llama1b_batched": llama1b_batched,
    "long_single": long_single,
    "skewed": skewed,
    "outliers": outliers,
}


def by_name(name: str, seed: int = 0) -> Workload:
    return NAMED[name](seed=seed)
