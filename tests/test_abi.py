"""CPU checks of the C-ABI boundary: the library loads, exports every entry point
include/flamia.h declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import precision_causal_attention_gb300 as F
    if not os.path.exists(F.LIB_PATH):
        from precision_causal_attention_gb300 import build
        build.build()
    return F.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "flamia.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(flamia_[a-z_]+)\s*\(", src)))


def test_header_declares_the_path_entry_points():
    names = declared_functions()
    for n in ("flamia_quantize", "flamia_fwd", "flamia_bwd", "flamia_get_status"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_sizes_are_host_computations(lib):
    import precision_causal_attention_gb300 as F
    T, Hq, Hkv, d = 1000, 4, 2, 64
    up = lambda x: (x + 255) // 256 * 256
    exp = 0
    for n in (T * Hq * d, T * Hkv * d, T * Hkv * d, T * Hq, T * Hkv, T * Hkv):
        exp = up(exp + n)
    # enough for every option: the common pieces, then the larger of the
    # NVFP4 pieces and the exact options' token-block V
    ext = max(up(T * Hq * d // 2) + up(T * Hkv * d // 2) + up(T * Hq * d // 16) + up(T * Hkv * d // 16),
              up(T * Hkv * d) + up(T * Hkv))
    assert F.flamia_saved_bytes(T, Hq, Hkv, d) == exp + ext
    assert F.flamia_saved_bytes_with(T, Hq, Hkv, d, F.default_opts()) == exp
    assert F.flamia_workspace_bytes(T, 3, Hq, Hkv, d) > T * Hq * d * 4
    assert F.flamia_saved_bytes(T, Hq, Hkv, 32) == 0          # unsupported d
    assert F.flamia_saved_bytes(T, 3, 2, 64) == 0             # Hq % Hkv != 0


def test_host_validation_rejects_before_launch(lib):
    import precision_causal_attention_gb300 as F
    vp = ctypes.c_void_p
    fake = vp(1 << 20)                      # never dereferenced: every case fails validation first
    o = F.default_opts()
    args = lambda d, opts, p=fake: (p, p, p, p, 3, 1000, 4, 2, d, ctypes.byref(opts), p, p, p, p, vp(0))
    assert lib.flamia_fwd(*args(32, o)) == -2
    assert lib.flamia_fwd(*args(96, o)) == -2
    bad = F.default_opts(c_exp=8, tau=2)    # c + tau > log2(448): the saturating setting of Appendix B.1
    assert lib.flamia_fwd(*args(64, bad)) == -1
    assert lib.flamia_fwd(*args(64, o, vp(0))) == -1          # null pointers
    assert lib.flamia_fwd(*args(64, o, vp((1 << 20) + 8))) == -3   # misaligned
    assert lib.flamia_quantize(fake, 1000, 4, 64, fake, -1, fake, fake, vp(0)) == -1
    assert lib.flamia_bwd(fake, fake, fake, fake, 3, 1000, 3, 2, 64, ctypes.byref(o), fake, fake, fake, fake, fake,
                          vp(0)) == -1
    rot = F.default_opts(hadamard=True)     # the rotation is defined for d = 128 only
    assert lib.flamia_fwd(*args(64, rot)) == -1
    assert lib.flamia_bwd(fake, fake, fake, fake, 3, 1000, 4, 2, 64, ctypes.byref(rot), fake, fake, fake, fake, fake,
                          vp(0)) == -1
    odd = F.default_opts()
    odd.hadamard = 2
    assert lib.flamia_fwd(*args(128, odd)) == -1
    odd = F.default_opts()
    odd.exact = 2
    assert lib.flamia_fwd(*args(64, odd)) == -1
    odd = F.default_opts()
    odd.schedule = 2                        # 0 dynamic hand-out, 1 static snake walk
    assert lib.flamia_fwd(*args(64, odd)) == -1
    ex = F.default_opts(exact=True)         # the score-tile dump serves token-block scales only
    assert lib.flamia_debug_set_score_dump(fake, fake, fake, fake, 0, 0, 0, 0) == 0
    try:
        assert lib.flamia_fwd(*args(64, ex)) == -7
        assert lib.flamia_bwd(fake, fake, fake, fake, 3, 1000, 4, 2, 128, ctypes.byref(ex), fake, fake, fake, fake,
                              fake, vp(0)) == -7
    finally:
        assert lib.flamia_debug_set_score_dump(None, None, None, None, 0, 0, 0, 0) == 0
    assert lib.flamia_debug_set_score_dump(fake, None, None, None, 0, 0, 0, 0) == -1   # pointers come in pairs
    assert lib.flamia_debug_set_item_limit(-1) == -1
    assert lib.flamia_debug_set_item_limit(0) == 0


def test_default_opts_are_the_mxfp8_setting(lib):
    import precision_causal_attention_gb300 as F
    o = F.default_opts()
    assert (o.c_exp, o.tau, o.causal, o.hadamard, o.exact, o.schedule) == (4, 4, 1, 0, 0, 0)
    assert F.default_opts(schedule="static").schedule == 1


def test_nvfp4_option_combinations_rejected(lib):
    import ctypes
    import precision_causal_attention_gb300 as F
    vp = ctypes.c_void_p
    fake = vp(1 << 20)
    args = lambda d, opts: (fake, fake, fake, fake, 3, 1000, 4, 2, d, ctypes.byref(opts), fake, fake, fake, fake, vp(0))
    assert lib.flamia_fwd(*args(64, F.default_opts(nvfp4=True, exact=True))) == -1
    assert lib.flamia_fwd(*args(128, F.default_opts(nvfp4=True, hadamard=True))) == -1
    odd = F.default_opts()
    odd.nvfp4 = 2
    assert lib.flamia_fwd(*args(64, odd)) == -1
    # the saved buffer grows by the NVFP4 Q and K
    T, Hq, Hkv, d = 1000, 4, 2, 64
    base = F.flamia_saved_bytes_with(T, Hq, Hkv, d, F.default_opts())
    up = lambda n: (n + 255) // 256 * 256
    extra = up(T * Hq * d // 2) + up(T * Hkv * d // 2) + up(T * Hq * d // 16) + up(T * Hkv * d // 16)
    assert F.flamia_saved_bytes_with(T, Hq, Hkv, d, F.default_opts(nvfp4=True)) == base + extra
    # the exact options add V with token-block scales
    extra_v = up(T * Hkv * d) + up(T * Hkv)
    assert F.flamia_saved_bytes_with(T, Hq, Hkv, d, F.default_opts(exact=True)) == base + extra_v
    # the size without options covers both
    assert F.flamia_saved_bytes(T, Hq, Hkv, d) == base + max(extra, extra_v)
    # the no-allocation forward leaves the NVFP4 path to flamia_fwd
    assert lib.flamia_fwd_noalloc(fake, fake, fake, fake, 3, 1000, 4, 2, 64, ctypes.byref(F.default_opts(nvfp4=True)),
                                  fake, fake, fake, vp(0)) == -7


def test_deterministic_dq_option_host_side(lib):
    import precision_causal_attention_gb300 as F
    vp = ctypes.c_void_p
    fake = vp(1 << 20)
    assert F.default_opts().deterministic_dq == 0
    assert F.default_opts(deterministic_dq=True).deterministic_dq == 1
    odd = F.default_opts()
    odd.deterministic_dq = 2
    args = lambda d, opts: (fake, fake, fake, fake, 3, 1000, 4, 2, d, ctypes.byref(opts), fake, fake, fake, fake,
                            fake, vp(0))
    assert lib.flamia_bwd(*args(64, odd)) == -1
    # not combined with the score-tile copy (a diagnostic of the fp32 path)
    det = F.default_opts(deterministic_dq=True)
    assert lib.flamia_debug_set_score_dump(fake, fake, fake, fake, 0, 0, 0, 0) == 0
    try:
        assert lib.flamia_bwd(*args(64, det)) == -7
    finally:
        assert lib.flamia_debug_set_score_dump(None, None, None, None, 0, 0, 0, 0) == 0
    # the workspace always has room for the 64-bit fixed-point accumulator
    T, Hq, Hkv, d = 1000, 4, 2, 64
    assert F.flamia_workspace_bytes(T, 3, Hq, Hkv, d) > T * Hq * d * 8
