"""flamia_fwd_noalloc: the forward for callers that cannot allocate device memory.

Such callers (code inside an allocator or memory-pool callback, runtimes that
only hand out pre-registered buffers, processes that reserve all device memory
up front) cannot provide flamia_fwd's workspace.  The no-allocation entry point
keeps the forward's work list in a fixed device array inside the library
instead.  This test calls it through the C ABI twice in a row, on two different
problems, and checks that each result is bitwise flamia_fwd's.  It lives in a file
collected last so that a run stopping at the first failure has run every other
test before it.
"""
import ctypes

import numpy as np
import pytest
import torch

import precision_causal_attention_gb300 as F
import workloads as W

pytestmark = pytest.mark.gpu


def _run_both(w):
    dev = torch.device("cuda:0")
    q, k, v = (w.tensors[n].to(dev) for n in ("q", "k", "v"))
    cu = torch.from_numpy(np.asarray(w.cu_seqlens, np.int32)).to(dev)
    T, Hq, Hkv, d = w.T, w.Hq, w.Hkv, w.d
    ref = F.Buffers(T, w.n_docs, Hq, Hkv, d)
    F.flamia_fwd(q, k, v, cu, ref.out, ref.lse, ref.saved, ref.work)
    out = torch.full((T, Hq, d), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((Hq, T), float("nan"), dtype=torch.float32, device=dev)
    saved = torch.zeros(F.flamia_saved_bytes(T, Hq, Hkv, d), dtype=torch.uint8, device=dev)
    o = F.default_opts()
    rc = F.lib().flamia_fwd_noalloc(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                                    ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(cu.data_ptr()), w.n_docs, T, Hq, Hkv,
                                    d, ctypes.byref(o), ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
                                    ctypes.c_void_p(saved.data_ptr()),
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    assert F.flamia_get_status() == 0
    return ref, out, lse, saved


def test_noalloc_forward_matches_flamia_fwd_twice_in_a_row():
    problems = [W.custom([300, 17, 129, 0, 256, 1, 40], Hq=4, Hkv=2, d=64, seed=11, T=800),
                W.custom([700, 90, 33], Hq=2, Hkv=1, d=128, seed=12)]
    for w in problems:
        ref, out, lse, saved = _run_both(w)
        # same plan, quantizer and forward kernel, and the forward has no
        # order-dependent sums: O and LSE must be the same bits (LSE is +inf
        # on both sides outside the documents)
        assert torch.isfinite(out.float()).all()
        assert torch.equal(out, ref.out)
        assert torch.equal(lse, ref.lse)
        # the quantized operands the backward would read are the same bytes
        va = F.saved_views(saved, w.T, w.Hq, w.Hkv, w.d)
        vb = F.saved_views(ref.saved, w.T, w.Hq, w.Hkv, w.d)
        for key in va:
            assert torch.equal(va[key], vb[key]), key


def test_noalloc_rejects_problems_beyond_its_limits():
    o = F.default_opts()
    vp = ctypes.c_void_p
    fake = vp(1 << 20)
    # more documents than the fixed work list holds: rejected before any launch
    rc = F.lib().flamia_fwd_noalloc(fake, fake, fake, fake, 65537, 1 << 17, 1, 1, 64, ctypes.byref(o), fake, fake, fake,
                                    vp(0))
    assert rc == -6
    rc = F.lib().flamia_fwd_noalloc(fake, fake, fake, fake, 1, (1 << 20) + 1, 1, 1, 64, ctypes.byref(o), fake, fake,
                                    fake, vp(0))
    assert rc == -6
