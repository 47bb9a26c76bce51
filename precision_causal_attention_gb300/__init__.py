"""Python binding of the flamia C ABI (include/flamia.h).

Argument marshalling only: every step of the attention path runs in the
CUDA kernels of ``libflamia_sm103.so``.  Tensors are torch CUDA tensors
(PyTorch supplies device memory and streams); each function passes their
device pointers and sizes to the C entry point of the same name and raises
``FlamiaError`` on a non-zero return code.  There is no CPU fallback: if the
library has not been built, every call fails loudly.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libflamia_sm103.so")

FLAMIA_STATUS = {0: "ok", 1: "bad cu_seqlens", 2: "on-chip wait timed out"}
ERRORS = {-1: "bad argument", -2: "unsupported head dimension", -3: "misaligned pointer",
          -4: "launch failed", -5: "unsupported device", -6: "beyond the no-allocation limits",
          -7: "option not implemented by this entry point"}


class FlamiaError(RuntimeError):
    pass


class Opts(ctypes.Structure):
    """flamia_opts: probability multiplier 2^c_exp, rescale threshold tau (log2 units), causal flag,
    Hadamard rotation of Q and K (d = 128), exact options (per-token scales), work hand-out
    (0 dynamic, 1 static snake walk), mixed NVFP4/FP8 path, order-independent (fixed-point) dQ."""
    _fields_ = [("c_exp", ctypes.c_int32), ("tau", ctypes.c_int32), ("causal", ctypes.c_int32),
                ("hadamard", ctypes.c_int32), ("exact", ctypes.c_int32), ("schedule", ctypes.c_int32),
                ("nvfp4", ctypes.c_int32), ("deterministic_dq", ctypes.c_int32)]


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise FlamiaError(f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        L.flamia_default_opts.restype = Opts
        L.flamia_saved_bytes.argtypes = [i64, i32, i32, i32]
        L.flamia_saved_bytes.restype = sz
        L.flamia_saved_bytes_with.argtypes = [i64, i32, i32, i32, ctypes.POINTER(Opts)]
        L.flamia_saved_bytes_with.restype = sz
        L.flamia_workspace_bytes.argtypes = [i64, i32, i32, i32, i32]
        L.flamia_workspace_bytes.restype = sz
        L.flamia_quantize.argtypes = [vp, i64, i32, i32, vp, i32, vp, vp, vp]
        L.flamia_quantize.restype = ctypes.c_int
        L.flamia_fwd.argtypes = [vp, vp, vp, vp, i32, i64, i32, i32, i32, ctypes.POINTER(Opts), vp, vp, vp, vp, vp]
        L.flamia_fwd.restype = ctypes.c_int
        L.flamia_bwd.argtypes = [vp, vp, vp, vp, i32, i64, i32, i32, i32, ctypes.POINTER(Opts), vp, vp, vp, vp, vp, vp]
        L.flamia_bwd.restype = ctypes.c_int
        L.flamia_fwd_noalloc.argtypes = [vp, vp, vp, vp, i32, i64, i32, i32, i32, ctypes.POINTER(Opts), vp, vp, vp,
                                         vp]
        L.flamia_fwd_noalloc.restype = ctypes.c_int
        L.flamia_get_status.argtypes = [ctypes.POINTER(i32), vp]
        L.flamia_get_status.restype = ctypes.c_int
        L.flamia_last_launch_count.restype = i32
        L.flamia_debug_set_score_dump.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32]
        L.flamia_debug_set_score_dump.restype = ctypes.c_int
        L.flamia_debug_set_item_limit.argtypes = [i32]
        L.flamia_debug_set_item_limit.restype = ctypes.c_int
        _lib = L
    return _lib


def _p(t: torch.Tensor) -> ctypes.c_void_p:
    if not t.is_cuda:
        raise FlamiaError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise FlamiaError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _s(stream: Optional[torch.cuda.Stream]) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(rc: int, what: str):
    if rc != 0:
        raise FlamiaError(f"{what}: {ERRORS.get(rc, rc)}")


def default_opts(causal: bool = True, c_exp: int = 4, tau: int = 4, hadamard: bool = False,
                 exact: bool = False, schedule: str = "dynamic", nvfp4: bool = False,
                 deterministic_dq: bool = False) -> Opts:
    if schedule not in ("dynamic", "static"):
        raise FlamiaError(f"schedule must be 'dynamic' or 'static', not {schedule!r}")
    o = lib().flamia_default_opts()
    o.causal, o.c_exp, o.tau, o.hadamard, o.exact = int(causal), int(c_exp), int(tau), int(hadamard), int(exact)
    o.schedule = 0 if schedule == "dynamic" else 1
    o.nvfp4 = int(nvfp4)
    o.deterministic_dq = int(deterministic_dq)
    return o


def flamia_saved_bytes(T: int, Hq: int, Hkv: int, d: int) -> int:
    return int(lib().flamia_saved_bytes(T, Hq, Hkv, d))


def flamia_saved_bytes_with(T: int, Hq: int, Hkv: int, d: int, opts: Opts) -> int:
    return int(lib().flamia_saved_bytes_with(T, Hq, Hkv, d, ctypes.byref(opts)))


def flamia_workspace_bytes(T: int, n_docs: int, Hq: int, Hkv: int, d: int) -> int:
    return int(lib().flamia_workspace_bytes(T, n_docs, Hq, Hkv, d))


def flamia_quantize(x: torch.Tensor, cu_seqlens: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor,
                    stream=None):
    """x bf16 [T,H,d] -> codes uint8 [T,H,d], scales uint8 [H,T] (document-local 32-token blocks)."""
    T, H, d = x.shape
    _check(lib().flamia_quantize(_p(x), T, H, d, _p(cu_seqlens), cu_seqlens.numel() - 1, _p(codes), _p(scales),
                                 _s(stream)), "flamia_quantize")


def flamia_fwd(q, k, v, cu_seqlens, out, lse, saved, work, opts: Optional[Opts] = None, stream=None):
    """MXFP8 forward: q [T,Hq,d], k/v [T,Hkv,d] bf16 -> out bf16 [T,Hq,d], lse fp32 [Hq,T]; fills `saved`."""
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    o = opts if opts is not None else default_opts()
    _check(lib().flamia_fwd(_p(q), _p(k), _p(v), _p(cu_seqlens), cu_seqlens.numel() - 1, T, Hq, Hkv, d,
                            ctypes.byref(o), _p(out), _p(lse), _p(saved), _p(work), _s(stream)), "flamia_fwd")


def flamia_fwd_noalloc(q, k, v, cu_seqlens, out, lse, saved, opts: Optional[Opts] = None, stream=None):
    """flamia_fwd without a workspace, for callers that cannot allocate (see include/flamia.h)."""
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    o = opts if opts is not None else default_opts()
    _check(lib().flamia_fwd_noalloc(_p(q), _p(k), _p(v), _p(cu_seqlens), cu_seqlens.numel() - 1, T, Hq, Hkv, d,
                                    ctypes.byref(o), _p(out), _p(lse), _p(saved), _s(stream)), "flamia_fwd_noalloc")


def flamia_bwd(out, lse, dout, cu_seqlens, saved, dq, dk, dv, work, opts: Optional[Opts] = None, stream=None):
    """MXFP8 backward from the forward's out, lse and saved codes: dout bf16 [T,Hq,d] -> dq, dk, dv bf16."""
    T, Hq, d = out.shape
    Hkv = dk.shape[1]
    o = opts if opts is not None else default_opts()
    _check(lib().flamia_bwd(_p(out), _p(lse), _p(dout), _p(cu_seqlens), cu_seqlens.numel() - 1, T, Hq, Hkv, d,
                            ctypes.byref(o), _p(saved), _p(dq), _p(dk), _p(dv), _p(work), _s(stream)), "flamia_bwd")


def flamia_get_status(stream=None) -> int:
    v = ctypes.c_int32(0)
    _check(lib().flamia_get_status(ctypes.byref(v), _s(stream)), "flamia_get_status")
    return int(v.value)


def flamia_last_launch_count() -> int:
    return int(lib().flamia_last_launch_count())


def flamia_debug_set_score_dump(s_fwd=None, f_fwd=None, s_bwd=None, f_bwd=None, h=0, doc=0, qt=0, kt=0):
    """Diagnostic hook: copy one score tile out of the forward and backward kernels (see include/flamia.h).
    Called with no tensors it switches the hook off."""
    ptr = lambda t: _p(t) if t is not None else ctypes.c_void_p(0)
    _check(lib().flamia_debug_set_score_dump(ptr(s_fwd), ptr(f_fwd), ptr(s_bwd), ptr(f_bwd), h, doc, qt, kt),
           "flamia_debug_set_score_dump")


def flamia_debug_set_item_limit(n: int) -> None:
    """Diagnostic: each forward CTA hands out at most n items (0 = off), so the call's waits time out."""
    _check(lib().flamia_debug_set_item_limit(int(n)), "flamia_debug_set_item_limit")


def saved_views(saved: torch.Tensor, T: int, Hq: int, Hkv: int, d: int, nvfp4: bool = False, exact: bool = False):
    """Views of the quantized Q, K, V inside the buffer flamia_fwd fills (layout of flamia_saved_bytes,
    and with nvfp4 the NVFP4 Q and K, with exact the token-block V copy, of flamia_saved_bytes_with)."""
    def up(x):
        return (x + 255) // 256 * 256
    o = 0
    out = {}
    pieces = [("q_codes", T * Hq * d, (T, Hq, d)), ("k_codes", T * Hkv * d, (T, Hkv, d)),
              ("v_codes", T * Hkv * d, (T, Hkv, d)), ("q_scales", T * Hq, (Hq, T)),
              ("k_scales", T * Hkv, (Hkv, T)), ("v_scales", T * Hkv, (Hkv, T))]
    if nvfp4:
        pieces += [("q4_codes", T * Hq * d // 2, (T, Hq, d // 2)), ("k4_codes", T * Hkv * d // 2, (T, Hkv, d // 2)),
                   ("q4_scales", T * Hq * d // 16, (T, Hq, d // 16)), ("k4_scales", T * Hkv * d // 16, (T, Hkv, d // 16))]
    if exact:
        pieces += [("vb_codes", T * Hkv * d, (T, Hkv, d)), ("vb_scales", T * Hkv, (Hkv, T))]
    for name, n, shape in pieces:
        out[name] = saved[o:o + n].view(shape)
        o = up(o + n)
    return out


def workspace_views(work: torch.Tensor, T: int, n_docs: int, Hq: int, d: int):
    """Views of the quantized dO, its scales and D inside the workspace after flamia_bwd."""
    def up(x):
        return (x + 255) // 256 * 256
    cap = (T + 127) // 128
    cvec = (cap + 2) * 4
    o = up(16)
    o = up(o + max(n_docs, 1) * 4)
    for _ in range(4):
        o = up(o + cvec)
    o = up(o + (cap + n_docs) * 16)          # item records
    out = {}
    out["do_codes"] = work[o:o + T * Hq * d].view(T, Hq, d); o = up(o + T * Hq * d)
    out["do_scales"] = work[o:o + T * Hq].view(Hq, T); o = up(o + T * Hq)
    out["D"] = work[o:o + T * Hq * 4].view(torch.float32).view(Hq, T)
    return out


class Buffers:
    """Caller-owned device buffers for one problem shape (allocated with torch)."""

    def __init__(self, T: int, n_docs: int, Hq: int, Hkv: int, d: int, device="cuda", opts: Optional[Opts] = None):
        n_saved = flamia_saved_bytes_with(T, Hq, Hkv, d, opts) if opts is not None else flamia_saved_bytes(T, Hq, Hkv, d)
        self.saved = torch.empty(n_saved, dtype=torch.uint8, device=device)
        self.work = torch.empty(flamia_workspace_bytes(T, n_docs, Hq, Hkv, d), dtype=torch.uint8, device=device)
        self.out = torch.empty(T, Hq, d, dtype=torch.bfloat16, device=device)
        self.lse = torch.empty(Hq, T, dtype=torch.float32, device=device)
        self.dq = torch.empty(T, Hq, d, dtype=torch.bfloat16, device=device)
        self.dk = torch.empty(T, Hkv, d, dtype=torch.bfloat16, device=device)
        self.dv = torch.empty(T, Hkv, d, dtype=torch.bfloat16, device=device)
