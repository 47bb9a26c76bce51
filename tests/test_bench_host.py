"""Host-side helpers of the benchmark (no GPU): the source digest that keeps
committed DRAM-traffic figures tied to the kernels they were measured on."""
import importlib.util
import os

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
_spec = importlib.util.spec_from_file_location("bench_host", os.path.join(ROOT, "bench.py"))
bench = importlib.util.module_from_spec(_spec)
_spec.loader.exec_module(bench)


def test_comments_and_whitespace_do_not_change_the_digest_input():
    a = 'int a = 1;  // first\n/* block\n comment */ float b = 2.f;\n'
    b = 'int a=1;\n\n    float b = 2.f; // reformatted, new comment\n'
    assert bench._code_only(a) == bench._code_only(b) == "inta=1;floatb=2.f;"


def test_code_and_string_literals_do_change_it():
    assert bench._code_only("int a = 1;") != bench._code_only("int a = 2;")
    # a comment marker inside a string literal is code
    assert bench._code_only('p("// x");') == 'p("// x");'
    assert bench._code_only('p("a\\"//b");') == 'p("a\\"//b");'



def test_clock_sampler_cleans_up_after_itself():
    c = bench.Clocks(0)
    path = c.path
    r = c.stop()
    assert set(r) >= {"sm_mhz", "sm_max_mhz", "reasons"}
    assert not os.path.exists(path)


def test_cpulist_parsing():
    from precision_causal_attention_gb300.host_pipeline import parse_cpulist
    assert parse_cpulist("0-3,8,10-11\n") == {0, 1, 2, 3, 8, 10, 11}
    assert parse_cpulist("5") == {5}
    assert parse_cpulist("") == set()


def test_composite_roofline_arithmetic():
    cu = [0, 96, 160, 256, 1280]
    T, Hq, Hkv, d = 1300, 8, 2, 64
    L = np.diff(np.asarray(cu, np.float64))
    pairs = bench.visible_pairs(cu, Hq)
    fwd_f, bwd_f = bench.attention_flops(cu, Hq, d)
    # the causal FLOP count takes L^2/2 pairs per document, the pair count L(L+1)/2
    assert pairs - fwd_f / (4 * d) == Hq * L.sum() / 2
    assert bench.visible_pairs(cu, Hq, causal=False) == Hq * (L * L).sum()
    c = bench.composite_roofline(cu, T, Hq, Hkv, d, True, fp8_tflops=4000.0, hbm_gbs=6000.0, sm_mhz=2000.0, n_sms=152)
    b = c["attn_bwd_bounds"]
    assert abs(b["tensor"] - bwd_f / 4000e12 * 1e3) < 1e-12
    assert abs(b["mufu"] - pairs / (32 * 152 * 2000e6) * 1e3) < 1e-12
    assert abs(c["attn_fwd_bounds"]["alu"] / c["attn_bwd_bounds"]["alu"] - 1.75 / 3.0) < 1e-12
    assert c["parts"]["attn_bwd"] == max(b.values())
    assert abs(c["ms"] - sum(c["parts"].values())) < 1e-12
    q, dq, f = bench.quant_bytes(T, Hq, Hkv, d)
    assert abs(c["parts"]["quant_qkv"] - q / 6000e9 * 1e3) < 1e-12


def test_fp8_peak_choice_follows_the_timed_region():
    peaks = {"bf16_tflops": 1976.9, "bf16_tflops_sustained": 1752.8}
    assert bench.fp8_peak_for(24.0, peaks) == (2 * 1976.9, "burst")
    assert bench.fp8_peak_for(4000.0, peaks) == (2 * 1752.8, "sustained")


def test_accuracy_report_of_the_oracle_sample():
    """The bench line's accuracy figures: cosines of the GPU's O, dQ, dK, dV to
    exact fp64 attention on the sample's complete documents.  Handing it the
    exact values themselves must give cosine 1, and the simulated oracle's
    cosines must sit in the 8-bit band below it."""
    import tempfile
    import numpy as np
    import workloads as W
    from oracle import exact as OX
    w = W.by_name("llama1b_packed", seed=0)
    cu = np.asarray(w.cu_seqlens, np.int64)
    end = 2048
    kf = cu[cu <= end]
    tf = int(kf[-1])
    g = w.Hq // w.Hkv
    x = {n: w.tensors[n][:tf].float().numpy().astype(np.float64) for n in ("q", "k", "v", "do")}
    q, k, v, do = x["q"][:, :g], x["k"][:, :1], x["v"][:, :1], x["do"][:, :g]
    O, _ = OX.forward(q, k, v, kf)
    dq, dk, dv = OX.backward(q, k, v, do, kf)
    npz = os.path.join(tempfile.mkdtemp(), "gpu.npz")
    np.savez(npz, out=O, dq=dq, dk=dk, dv=dv)
    cb = bench.cpu_oracle_sample("llama1b_packed", rows_tokens=end, gpu_npz=npz)
    ac = cb["accuracy"]
    assert ac["tokens"] == tf
    for n in ("O", "dQ", "dK", "dV"):
        assert abs(ac["gpu_cosine"][n] - 1.0) < 1e-12, n
        assert 0.99 < ac["oracle_cosine"][n] < 1.0, n
