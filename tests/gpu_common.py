"""Helpers shared by the GPU tests: run the CUDA path through the C-ABI binding and
compare it with the oracle.  Only tests import this module."""
from __future__ import annotations

import numpy as np
import torch

import precision_causal_attention_gb300 as F


def rel_fro(a, b) -> float:
    a = np.asarray(a, np.float64); b = np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / den) if den > 0 else float(np.linalg.norm(a - b))


def cosine(a, b) -> float:
    a = np.asarray(a, np.float64).ravel(); b = np.asarray(b, np.float64).ravel()
    return float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b)))


def run_gpu(w, causal=True, do_bwd=True, tensors=None, c_exp=4, tau=4, hadamard=False, exact=False, nvfp4=False,
            deterministic_dq=False, schedule="dynamic"):
    """Run quantize + forward (+ backward) on cuda:0; returns CPU results."""
    dev = torch.device("cuda:0")
    t = tensors if tensors is not None else w.tensors
    q, k, v, do = (t[n].to(dev) for n in ("q", "k", "v", "do"))
    cu = torch.from_numpy(np.asarray(w.cu_seqlens, np.int32)).to(dev)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    opts = F.default_opts(causal=causal, c_exp=c_exp, tau=tau, hadamard=hadamard, exact=exact, nvfp4=nvfp4,
                          deterministic_dq=deterministic_dq, schedule=schedule)
    B = F.Buffers(T, w.n_docs, Hq, Hkv, d, opts=opts)
    # poison outputs so unwritten elements show up
    B.out.fill_(float("nan")); B.lse.fill_(float("nan"))
    B.dq.fill_(float("nan")); B.dk.fill_(float("nan")); B.dv.fill_(float("nan"))
    F.flamia_fwd(q, k, v, cu, B.out, B.lse, B.saved, B.work, opts)
    res = {}
    if do_bwd:
        F.flamia_bwd(B.out, B.lse, do, cu, B.saved, B.dq, B.dk, B.dv, B.work, opts)
    torch.cuda.synchronize()
    res["status"] = F.flamia_get_status()
    res["out"] = B.out.float().cpu().numpy().astype(np.float64)
    res["lse"] = B.lse.cpu().numpy().astype(np.float64)
    sv = F.saved_views(B.saved, T, Hq, Hkv, d, nvfp4=nvfp4, exact=exact)
    for kname in sv:
        res[kname] = sv[kname].cpu().numpy()
    if do_bwd:
        res["dq"] = B.dq.float().cpu().numpy().astype(np.float64)
        res["dk"] = B.dk.float().cpu().numpy().astype(np.float64)
        res["dv"] = B.dv.float().cpu().numpy().astype(np.float64)
        wv = F.workspace_views(B.work, T, w.n_docs, Hq, d)
        res["do_codes"] = wv["do_codes"].cpu().numpy()
        res["do_scales"] = wv["do_scales"].cpu().numpy()
        res["D"] = wv["D"].cpu().numpy().astype(np.float64)
    return res


def np_inputs(w, tensors=None):
    t = tensors if tensors is not None else w.tensors
    return {n: t[n].float().numpy().astype(np.float64) for n in ("q", "k", "v", "do")}
