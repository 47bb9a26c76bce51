#!/usr/bin/env python
"""Benchmark of the MXFP8 causal packed attention training call on GB300.

One step = the whole hot path on one batch of packed documents:
quantize Q/K/V -> forward -> quantize dO (+ D, dQ accumulator init) -> backward
(flamia_fwd + flamia_bwd, five kernel launches), inputs resident in HBM.

Metric: fwd+bwd attention TFLOP/s including quantization, with the causal
FLOP discount of the FLAMIA paper (Appendix E): forward = 4 Hq d sum_r L_r^2 / 2,
backward = 2.5 x forward.  Also reported as a fraction of the dense FP8 tensor
peak.  Workload (default): 4 rows x 8192 tokens of lognormal(median 1024, sigma 1)
documents in [32, 8192], 32 query / 8 key-value heads, d = 64, causal.

Timing: W untimed warm-up steps, then K steps, each bracketed by CUDA events on
the launching stream, with the 129 MB L2 flushed (a 512 MB write) between steps
outside the timed events.  Per-kernel times come from events the library records
around each of its launches.  Under torchrun each rank runs its own replica
(its own documents, same shape): the job total is N x one replica's work over the
slowest rank's time.

--impl reference times the CPU oracle (the only other implementation of the
method here) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 2.0        # nominal dense ratio (4.5 / 2.25 PFLOP/s)
METRIC = "fwd+bwd attention TFLOP/s incl. quantization (MXFP8, 1 GB300), % of FP8 peak"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


# Source files each timed kernel is compiled from.  profiles/traffic.json
# holds DRAM bytes per launch from an ncu capture together with a digest of
# these files; the figure is reported only while the digest still matches.
KERNEL_SOURCES = {
    "attn_bwd": ["bwd.cu", "bwd_d64.cu", "bwd_common.cuh", "flamia_common.cuh", "sm103_ptx.cuh", "launch.h"],
    "attn_fwd": ["fwd.cu", "flamia_common.cuh", "sm103_ptx.cuh", "launch.h"],
    "quant_qkv": ["prep.cu", "flamia_common.cuh", "sm103_ptx.cuh", "launch.h"],
    "quant_do": ["prep.cu", "flamia_common.cuh", "sm103_ptx.cuh", "launch.h"],
    "finalize_bwd": ["prep.cu", "flamia_common.cuh", "sm103_ptx.cuh", "launch.h"],
}


def _code_only(src: str) -> str:
    """C++ source without comments and whitespace (string literals kept), so
    that a comment edit does not count as a kernel change."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif c == '"':
            j = i + 1
            while j < n and src[j] != '"':
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        else:
            if not c.isspace():
                out.append(c)
            i += 1
    return "".join(out)


def kernel_source_digest(kernel: str) -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "precision_causal_attention_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        path = os.path.join(csrc, f)
        h.update(f.encode())
        h.update(_code_only(open(path).read()).encode() if os.path.exists(path) else b"<absent>")
    return h.hexdigest()[:16]


def measured_traffic(workload: str):
    """DRAM bytes per launch per kernel, for kernels whose sources are unchanged since the capture."""
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(tpath):
        return {}
    tj = json.load(open(tpath))
    if tj.get("workload") != workload:
        return {}
    return {k: v["bytes"] for k, v in tj.get("kernels", {}).items()
            if k in KERNEL_SOURCES and v.get("source_digest") == kernel_source_digest(k)}


def attention_flops(cu, Hq, d, causal=True):
    L = np.diff(np.asarray(cu, np.int64)).astype(np.float64)
    s2 = float((L * L).sum())
    fwd = 4.0 * Hq * d * (s2 / 2.0 if causal else s2)
    return fwd, 2.5 * fwd


def quant_bytes(T, Hq, Hkv, d):
    """Algorithmic bytes of the two quantizer passes and of the dQ finalisation.
    At d = 64 the forward clears the fp32 dQ accumulator (so the dO pass does
    not); at d = 128 the dO pass does."""
    n_qkv = T * (Hq + 2 * Hkv)
    qkv = n_qkv * d * 2 + n_qkv * d + n_qkv                       # read bf16, write codes + scales
    do = T * Hq * d * 2 * 2 + T * Hq * d + T * Hq + 4 * T * Hq   # dO, O in; codes, scales, D out
    if d != 64:
        do += 4 * T * Hq * d                                      # dQ accumulator cleared here
    fin = 4 * T * Hq * d + 2 * T * Hq * d                         # fp32 dQ in, bf16 dQ out
    return qkv, do, fin


# Rates of the composite roofline, per SM and clock (the clock is the median
# SM clock sampled during the timed region):
#   MUFU ex2: 32 results (the pages' figure for sm_103, twice sm_100's);
#   FP32 pipe: 128 lanes, an f32x2 instruction doing two elements per lane.
MUFU_PER_CLK_SM = 32
FP32_LANES_PER_CLK_SM = 128
# FP32-pipe lane slots per visible (query, key) pair, counted from the score
# arithmetic the kernels must do (packed f32x2 forms count half):
#   forward: scale-and-subtract (FFMA2, 1/2), row maximum (3-input max, 1/2),
#            row sum (FADD2, 1/2), E4M3 conversion (4 per instruction, 1/4);
#   backward: P argument (FFMA2, 1/2), dP - D (FFMA2, 1/2), dS = P (dP - D)
#            (FMUL2, 1/2), |dS| block maximum (1/2), dS scaling (1/2), P' and
#            dS conversions (2 x 1/4).
ALU_SLOTS_FWD = 1.75
ALU_SLOTS_BWD = 3.0


def visible_pairs(cu_seqlens, Hq, causal=True):
    """(query, key) pairs the attention visits, summed over query heads."""
    L = np.diff(np.asarray(cu_seqlens, np.int64)).astype(np.float64)
    return float(Hq * ((L * (L + 1) / 2).sum() if causal else (L * L).sum()))


def composite_roofline(cu_seqlens, T, Hq, Hkv, d, causal, fp8_tflops, hbm_gbs, sm_mhz, n_sms):
    """Lower bound on one step's time: the HBM-bound kernels at the copy
    bandwidth, plus for each attention kernel the largest of its tensor,
    MUFU, FP32-pipe and HBM times.  Returns per-kernel floors (ms)."""
    fwd_f, bwd_f = attention_flops(cu_seqlens, Hq, d, causal=causal)
    pairs = visible_pairs(cu_seqlens, Hq, causal)
    clk = sm_mhz * 1e6
    mufu_rate = MUFU_PER_CLK_SM * n_sms * clk
    alu_rate = FP32_LANES_PER_CLK_SM * n_sms * clk
    bw = hbm_gbs * 1e9
    qkv_b, do_b, fin_b = quant_bytes(T, Hq, Hkv, d)
    codes = T * (Hq + 2 * Hkv) * d + T * (Hq + 2 * Hkv)            # E4M3 codes + scale bytes
    fwd_b = codes + 2 * T * Hq * d + 4 * T * Hq + (4 * T * Hq * d if d == 64 else 0)
    bwd_b = codes + T * Hq * (d + 1) + 8 * T * Hq + 4 * T * Hkv * d + 4 * T * Hq * d
    ms = lambda sec: sec * 1e3
    fwd = {"tensor": ms(fwd_f / (fp8_tflops * 1e12)), "mufu": ms(pairs / mufu_rate),
           "alu": ms(ALU_SLOTS_FWD * pairs / alu_rate), "hbm": ms(fwd_b / bw)}
    bwd = {"tensor": ms(bwd_f / (fp8_tflops * 1e12)), "mufu": ms(pairs / mufu_rate),
           "alu": ms(ALU_SLOTS_BWD * pairs / alu_rate), "hbm": ms(bwd_b / bw)}
    parts = {"quant_qkv": ms(qkv_b / bw), "quant_do": ms(do_b / bw), "finalize_bwd": ms(fin_b / bw),
             "attn_fwd": max(fwd.values()), "attn_bwd": max(bwd.values())}
    return {"ms": sum(parts.values()), "parts": parts,
            "attn_fwd_bounds": fwd, "attn_bwd_bounds": bwd,
            "attn_fwd_bound": max(fwd, key=fwd.get), "attn_bwd_bound": max(bwd, key=bwd.get),
            "rates": {"fp8_tflops": fp8_tflops, "hbm_gbs": hbm_gbs, "sm_mhz": sm_mhz, "sms": n_sms,
                      "mufu_ex2_per_clk_sm": MUFU_PER_CLK_SM, "fp32_lanes_per_clk_sm": FP32_LANES_PER_CLK_SM,
                      "fp32_slots_per_pair": {"fwd": ALU_SLOTS_FWD, "bwd": ALU_SLOTS_BWD}},
            "visible_pairs": pairs}


def fp8_peak_for(timed_ms, peaks):
    """Dense FP8 denominator: the burst figure for a timed region under a
    second (the GPU does not reach its power-capped steady state), the
    sustained one otherwise; each is the bf16 figure x the nominal ratio."""
    if timed_ms < 1000.0:
        return peaks["bf16_tflops"] * FP8_OVER_BF16, "burst"
    return peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) * FP8_OVER_BF16, "sustained"


class Clocks:
    """nvidia-smi sampler for the timed region."""

    def __init__(self, gpu_index: int):
        import tempfile
        self.proc = None
        fd, self.path = tempfile.mkstemp(prefix=f"flamia_clocks_gpu{gpu_index}_", suffix=".csv")
        self.fh = os.fdopen(fd, "w")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index),
                 "--query-gpu=index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            self.fh.close()
            os.remove(self.path)
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.remove(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_oracle_sample(name: str, seed: int = 0, rows_tokens: int = 16384, steps: int = 1, timeout: int = 900,
                      causal: bool = True, gpu_npz: str = ""):
    """Time the oracle (quantize + simulated fwd + bwd) on the first `rows_tokens`
    packed tokens and one grouped-query group, `steps` times, in a fresh process
    (spawned, never forked after CUDA) with BLAS threads = host cores.

    gpu_npz: the GPU's O, dQ, dK, dV of that group on the sample's complete
    documents (arrays "out", "dq", "dk", "dv"); the process then also reports
    their cosines to exact fp64 attention (the oracle's unquantized reference)
    next to the simulated oracle's, on the same rows."""
    code = f"""
import json, os, sys, time
sys.path.insert(0, {ROOT!r})
import numpy as np
import workloads as W
from oracle import simulated as OS
w = W.by_name({name!r}, seed={seed})
cu = np.asarray(w.cu_seqlens, np.int64)
end = {rows_tokens}
keep = cu[cu <= end]
if keep[-1] != end:
    keep = np.append(keep, end)
Tn = int(keep[-1])
g = w.Hq // w.Hkv
x = {{n: w.tensors[n][:Tn].float().numpy().astype(np.float64) for n in ("q", "k", "v", "do")}}
q = x["q"][:, :g]; k = x["k"][:, :1]; v = x["v"][:, :1]; do = x["do"][:, :g]
secs = []
for _ in range({steps}):
    t0 = time.perf_counter()
    f = OS.forward(q, k, v, keep, causal={causal!r})
    b = OS.backward(q, k, v, f["O_bf16"], f["lse"], do, keep, causal={causal!r})
    secs.append(time.perf_counter() - t0)
L = np.diff(keep).astype(np.float64)
fwd = 4.0 * g * w.d * float((L * L).sum()) / ({2.0 if causal else 1.0})
res = {{"seconds": secs, "flops": 3.5 * fwd, "tokens": Tn, "heads": g, "docs": int(len(keep) - 1)}}
if {gpu_npz!r}:
    from oracle import exact as OX
    z = np.load({gpu_npz!r})
    kf = cu[cu <= end]
    Tf = int(kf[-1])
    Ox, _ = OX.forward(q[:Tf], k[:Tf], v[:Tf], kf, causal={causal!r})
    gx = OX.backward(q[:Tf], k[:Tf], v[:Tf], do[:Tf], kf, causal={causal!r})
    fs = OS.forward(q[:Tf], k[:Tf], v[:Tf], kf, causal={causal!r})
    bs = OS.backward(q[:Tf], k[:Tf], v[:Tf], fs["O_bf16"], fs["lse"], do[:Tf], kf, causal={causal!r})
    def cosine(a, b):
        a = np.asarray(a, np.float64).ravel(); b = np.asarray(b, np.float64).ravel()
        return float(a @ b / np.sqrt((a @ a) * (b @ b)))
    ref = {{"O": Ox, "dQ": gx[0], "dK": gx[1], "dV": gx[2]}}
    gpu = {{"O": z["out"], "dQ": z["dq"], "dK": z["dk"], "dV": z["dv"]}}
    sim = {{"O": fs["O"], "dQ": bs["dq"], "dK": bs["dk"], "dV": bs["dv"]}}
    res["accuracy"] = {{"tokens": Tf, "docs": int(len(kf) - 1),
                        "gpu_cosine": {{n: cosine(gpu[n], ref[n]) for n in ref}},
                        "oracle_cosine": {{n: cosine(sim[n], ref[n]) for n in ref}}}}
print(json.dumps(res))
"""
    ncpu = os.cpu_count() or 1
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = str(ncpu)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=timeout)
    if r.returncode != 0:
        raise RuntimeError("oracle sample failed: " + r.stderr[-2000:])
    out = json.loads(r.stdout.strip().splitlines()[-1])
    out["cores"] = ncpu
    return out


def sample_desc(cb):
    return (f"first {cb['tokens']} packed tokens ({cb['docs']} documents), one grouped-query group "
            f"({cb['heads']} query heads, 1 KV head): token-block quantize + simulated fwd + bwd")


def run_reference(args):
    from precision_causal_attention_gb300.replicas import rank_env
    if rank_env().rank != 0:
        return 0
    import workloads as W
    w = W.by_name(args.workload, seed=0)
    # one step = one bounded sample; a smaller sample when many steps are asked,
    # so the whole run stays within a few minutes
    tokens = 8192 if args.steps <= 24 else 2048
    cb = cpu_oracle_sample(args.workload, rows_tokens=tokens, steps=args.steps + args.warmup,
                           causal=not args.noncausal)
    secs = cb["seconds"][args.warmup:]
    value = cb["flops"] * len(secs) / sum(secs) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": int(args.gpus),
        "steps": len(secs), "warmup": args.warmup, "ms_per_step": 1e3 * sum(secs) / len(secs),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d, "causal": not args.noncausal},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cb["cores"], "kind": "oracle",
                         "sample": sample_desc(cb)},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch
    import precision_causal_attention_gb300 as F
    import workloads as W

    from precision_causal_attention_gb300.replicas import rank_env, max_over_ranks, whole_job_rate
    env = rank_env()
    world, rank, local = env.world, env.rank, env.local
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    w = W.by_name(args.workload, seed=rank)           # each replica: its own documents, same shape
    T, Hq, Hkv, d = w.T, w.Hq, w.Hkv, w.d
    q, k, v, do = (w.tensors[n].to(dev) for n in ("q", "k", "v", "do"))
    cu = torch.from_numpy(np.asarray(w.cu_seqlens, np.int32)).to(dev)
    causal = not args.noncausal
    opts = F.default_opts(causal=causal, exact=args.exact, schedule=args.schedule, nvfp4=args.nvfp4,
                          deterministic_dq=args.deterministic_dq)
    B = F.Buffers(T, w.n_docs, Hq, Hkv, d, device=dev, opts=opts)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    # per-launch events recorded by the library: before each launch and after
    # the last (the forward makes 2 launches, the backward 3)
    # the exact options add a launch that keeps a token-block copy of V
    FWD_KERNELS = ("quant_qkv", "quant_vb", "attn_fwd") if args.exact else ("quant_qkv", "attn_fwd")
    BWD_KERNELS = ("quant_do", "attn_bwd", "finalize_bwd")
    ev_f = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    for e in ev_f + ev_b:
        e.record(stream)                               # torch creates events lazily
    torch.cuda.synchronize(dev)
    import ctypes
    arr_f = (ctypes.c_void_p * 5)(*[e.cuda_event for e in ev_f])
    arr_b = (ctypes.c_void_p * 5)(*[e.cuda_event for e in ev_b])
    L = F.lib()

    def step(hooks: bool):
        if hooks:
            L.flamia_set_launch_events(arr_f, 5)
        F.flamia_fwd(q, k, v, cu, B.out, B.lse, B.saved, B.work, opts)
        if hooks:
            L.flamia_set_launch_events(arr_b, 5)
        F.flamia_bwd(B.out, B.lse, do, cu, B.saved, B.dq, B.dk, B.dv, B.work, opts)
        if hooks:
            L.flamia_set_launch_events(None, 0)

    for _ in range(args.warmup):
        step(False)
    torch.cuda.synchronize(dev)
    status = F.flamia_get_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after warm-up")

    # The whole step (5 launches) is captured once into a CUDA graph and
    # replayed: the library's calls allocate nothing and never synchronise, so
    # they are capture-safe; the per-launch timing events are captured with
    # them and recorded on every replay.
    graph, graph_note = None, "off (--no-graph)"
    if not args.no_graph:
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step(True)
            graph, graph_note = g, "one CUDA graph per step"
        except Exception as e:  # keep measuring without it, and say so
            graph_note = f"capture failed: {e}"[:160]
            torch.cuda.synchronize(dev)
        L.flamia_set_launch_events(None, 0)

    def run_step(hooks: bool):
        if graph is not None:
            graph.replay()
        else:
            step(hooks)

    for _ in range(2):                                 # first replays outside the timed region
        run_step(False)
    torch.cuda.synchronize(dev)

    clk = Clocks(local)
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    step_ms, kern = [], {n: [] for n in FWD_KERNELS + BWD_KERNELS}
    t_wall0 = time.perf_counter()
    for _ in range(args.steps):
        flush.zero_()
        s0 = torch.cuda.Event(enable_timing=True); s1 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        run_step(True)
        s1.record(stream)
        s1.synchronize()
        step_ms.append(s0.elapsed_time(s1))
        for i, n in enumerate(FWD_KERNELS):
            kern[n].append(ev_f[i].elapsed_time(ev_f[i + 1]))
        for i, n in enumerate(BWD_KERNELS):
            kern[n].append(ev_b[i].elapsed_time(ev_b[i + 1]))
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - t_wall0
    if dist:
        dist.barrier()
    clocks = clk.stop()
    status = F.flamia_get_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed steps")

    total_ms = max_over_ranks(float(sum(step_ms)), dist, dev)
    fwd_f, bwd_f = attention_flops(w.cu_seqlens, Hq, d, causal=causal)
    step_flops = fwd_f + bwd_f
    value = whole_job_rate(world, step_flops, args.steps, total_ms) / 1e12
    ms_per_step = total_ms / args.steps

    # ---------------- end to end through the C-ABI with host buffers
    # Every step copies its inputs from pinned host memory to the device and
    # its results back; the pipeline keeps two steps in flight, so step i+1's
    # inputs and step i-1's results travel while step i computes.
    from precision_causal_attention_gb300.host_pipeline import HostPipeline, bind_to_gpu_node
    # pinned buffers allocated (and first touched) from the GPU's NUMA node;
    # the process's CPU set is restored afterwards
    aff = os.sched_getaffinity(0) if hasattr(os, "sched_getaffinity") else None
    numa_bound = bind_to_gpu_node(dev)
    hin = {n: w.tensors[n].pin_memory() for n in ("q", "k", "v", "do")}
    hin["cu"] = torch.from_numpy(np.asarray(w.cu_seqlens, np.int32)).pin_memory()
    houts = [{n: torch.zeros(getattr(B, n).shape, dtype=getattr(B, n).dtype).pin_memory()
              for n in ("out", "lse", "dq", "dk", "dv")} for _ in range(2)]
    if numa_bound and aff is not None:
        os.sched_setaffinity(0, aff)
    h2d, d2h = HostPipeline.bytes_per_batch(hin, houts[0])
    pipe = HostPipeline(T, w.n_docs, Hq, Hkv, d, device=dev, opts=opts, pre_step=flush.zero_)
    for i in range(args.warmup):
        pipe.submit(hin, houts[i % 2])
    pipe.synchronize()
    if F.flamia_get_status() != 0:
        raise RuntimeError("device status after the end-to-end warm-up")
    if dist:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True); e1 = torch.cuda.Event(enable_timing=True)
    e0.record(pipe.copy_in_stream)
    for i in range(args.steps):
        pipe.submit(hin, houts[i % 2])
    e1.record(pipe.copy_out_stream)
    pipe.synchronize()
    e2e_total = float(e0.elapsed_time(e1))
    if F.flamia_get_status() != 0:
        raise RuntimeError("device status after the end-to-end steps")
    e2e_total = max_over_ranks(e2e_total, dist, dev)
    e2e_value = whole_job_rate(world, step_flops, args.steps, e2e_total) / 1e12

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    peaks, peak_src = load_peaks()
    fp8_peak, fp8_kind = fp8_peak_for(total_ms, peaks)
    sm_mhz = clocks.get("sm_mhz") or peaks.get("sm_max_mhz") or 2070.0
    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    comp = composite_roofline(w.cu_seqlens, T, Hq, Hkv, d, causal, fp8_peak, peaks["hbm_gbs"], sm_mhz, n_sms)
    comp["frac"] = comp["ms"] / ms_per_step
    km = {n: statistics.mean(v) for n, v in kern.items()}
    qkv_b, do_b, fin_b = quant_bytes(T, Hq, Hkv, d)
    kernels = {
        "attn_bwd": {"ms": km["attn_bwd"], "bound": "tensor", "achieved": bwd_f / (km["attn_bwd"] * 1e-3) / 1e12,
                     "unit": "TFLOP/s", "peak": fp8_peak},
        "attn_fwd": {"ms": km["attn_fwd"], "bound": "tensor", "achieved": fwd_f / (km["attn_fwd"] * 1e-3) / 1e12,
                     "unit": "TFLOP/s", "peak": fp8_peak},
        "quant_qkv": {"ms": km["quant_qkv"], "bound": "hbm", "achieved": qkv_b / (km["quant_qkv"] * 1e-3) / 1e9,
                      "unit": "GB/s", "peak": peaks["hbm_gbs"]},
        "quant_do": {"ms": km["quant_do"], "bound": "hbm", "achieved": do_b / (km["quant_do"] * 1e-3) / 1e9,
                     "unit": "GB/s", "peak": peaks["hbm_gbs"]},
        "finalize_bwd": {"ms": km["finalize_bwd"], "bound": "hbm", "achieved": fin_b / (km["finalize_bwd"] * 1e-3) / 1e9,
                         "unit": "GB/s", "peak": peaks["hbm_gbs"]},
    }
    if "quant_vb" in km:
        # V read (bf16) + codes + one scale byte per token-head
        vb_b = T * Hkv * d * 2 + T * Hkv * d + T * Hkv
        kernels["quant_vb"] = {"ms": km["quant_vb"], "bound": "hbm", "achieved": vb_b / (km["quant_vb"] * 1e-3) / 1e9,
                               "unit": "GB/s", "peak": peaks["hbm_gbs"]}
    for kk in kernels.values():
        if "achieved" in kk:
            kk["frac"] = kk["achieved"] / kk["peak"]
    dom = max(("attn_bwd", "attn_fwd", "quant_qkv", "quant_do"), key=lambda n: kernels[n]["ms"])
    measured = measured_traffic(w.name)
    for n, kk in kernels.items():
        if "achieved" in kk:
            kk["traffic"] = measured.get(n)
    traffic = measured.get(dom)
    dk = kernels[dom]
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
        "fp8_peak_frac": value / world / fp8_peak,
        "fp8_peak_tflops": fp8_peak,
        "fp8_peak_source": (f"{peak_src} bf16 {fp8_kind} x{FP8_OVER_BF16:g} (nominal dense FP8/BF16 ratio); "
                            f"{fp8_kind}: timed region {total_ms:.0f} ms"),
        "composite_roofline": comp,
        "config": {"workload": w.name, "T": T, "Hq": Hq, "Hkv": Hkv, "d": d, "causal": causal,
                   **({"exact_options": True} if args.exact else {}),
                   **({"scores": "nvfp4 (mixed NVFP4/FP8 path)"} if args.nvfp4 else {}),
                   **({"dq_accumulation": "64-bit fixed point (order-independent)"} if args.deterministic_dq else {}),
                   "schedule": args.schedule,
                   "n_docs": w.n_docs, "max_doc": int(np.diff(w.cu_seqlens).max()),
                   "flops_per_step": step_flops, "l2": "flushed (512 MB write) between timed steps",
                   "launch": graph_note,
                   "parallelism": "replicas" if world > 1 else "single"},
        "roofline": {"kernel": dom, "bound": dk["bound"], "achieved": dk["achieved"], "peak": dk["peak"],
                     "unit": dk["unit"], "frac": dk["frac"], "traffic": traffic,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json)" + (f", fp8 = bf16 {fp8_kind} x2" if dk["bound"] == "tensor" else "")},
        "kernels": kernels,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "ms_per_step": e2e_total / args.steps,
                "launch": "eager, two steps in flight: copies on two streams overlap the kernels (HostPipeline)",
                "host_buffers": "pinned on the GPU's NUMA node" if numa_bound else "pinned (NUMA node not found)"},
        "gpu_launches": (len(FWD_KERNELS) + len(BWD_KERNELS)) * args.steps,
        "clocks": clocks,
        "wall_s": wall,
    }
    if not args.no_cpu_baseline:
        try:
            # the GPU's results for the oracle sample's complete documents and
            # first grouped-query group, for the accuracy figures
            import tempfile
            cuv = np.asarray(w.cu_seqlens, np.int64)
            tf = int(cuv[cuv <= 16384][-1])
            g = Hq // Hkv
            npz = os.path.join(tempfile.mkdtemp(prefix="flamia_acc_"), "gpu.npz")
            np.savez(npz, out=B.out[:tf, :g].float().cpu().numpy(), dq=B.dq[:tf, :g].float().cpu().numpy(),
                     dk=B.dk[:tf, :1].float().cpu().numpy(), dv=B.dv[:tf, :1].float().cpu().numpy())
            cb = cpu_oracle_sample(args.workload, causal=causal, gpu_npz=npz)
            line["cpu_baseline"] = {
                "value": cb["flops"] / cb["seconds"][0] / 1e12, "unit": "TFLOP/s", "cores": cb["cores"],
                "kind": "oracle", "sample": sample_desc(cb) + f", {cb['seconds'][0]:.1f} s"}
            if "accuracy" in cb:
                ac = cb["accuracy"]
                line["accuracy"] = {
                    "vs": "exact fp64 attention (the oracle's unquantized reference)",
                    "sample": (f"first {ac['tokens']} packed tokens ({ac['docs']} complete documents), "
                               f"query heads 0..{g - 1} and KV head 0"),
                    "gpu_cosine": ac["gpu_cosine"],
                    "oracle_cosine": ac["oracle_cosine"] if not (args.exact or args.nvfp4) else
                    "(token-block oracle; the option's own oracle is in the tests)"}
        except Exception as e:  # the GPU line must still print
            line["cpu_baseline"] = {"value": None, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                                    "sample": f"failed: {e}"[:200]}
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="llama1b_packed")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch the 5 kernels per step without a CUDA graph")
    ap.add_argument("--schedule", choices=("dynamic", "static"), default="dynamic",
                    help="work hand-out of the attention kernels: run-time claims (default) or the static snake walk")
    ap.add_argument("--nvfp4", action="store_true",
                    help="the mixed NVFP4/FP8 path (4-bit Q and K for the scores, log-domain P-hat)")
    ap.add_argument("--exact", action="store_true",
                    help="the exact options (per-token scales and folded payloads)")
    ap.add_argument("--deterministic-dq", action="store_true",
                    help="order-independent dQ: 64-bit fixed-point partials added with integer reduce-adds")
    ap.add_argument("--noncausal", action="store_true",
                    help="full attention within each document (the headline line is causal); FLOPs without the causal discount")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
