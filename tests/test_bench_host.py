"""Host-side helpers of the benchmark (no GPU): the source digest that keeps
committed DRAM-traffic figures tied to the kernels they were measured on."""
import importlib.util
import os

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
