"""Multi-process host logic on CPU: two gloo ranks run as replicas (each its
own batch of the same shape), share only their timing, and agree on the
slowest rank's time and the whole-job rate.  The reference arm prints from
rank 0 only."""
import os
import socket
import types

import numpy as np
import pytest

from precision_causal_attention_gb300.replicas import max_over_ranks, rank_env, whole_job_rate


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _replica(rank, world, port, out):
    import torch.distributed as dist
    import workloads as W
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    env = rank_env()
    dist.init_process_group("gloo", rank=env.rank, world_size=env.world)
    try:
        w = W.llama1b_packed(seed=env.rank, rows=1, row_len=2048)   # the bench seeds each replica by rank
        mine = 100.0 + 37.5 * env.rank                              # this rank's timed total, ms
        slow = max_over_ranks(mine, dist)
        rate = whole_job_rate(env.world, 1.0e12, 10, slow)
        dist.barrier()
        out.put((env.rank, slow, rate, tuple(w.tensors["q"].shape), list(np.asarray(w.cu_seqlens))))
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas_share_only_the_slowest_time():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_replica, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = sorted(out.get(timeout=180) for _ in range(2))
    finally:
        for p in procs:
            p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs)
    (r0, slow0, rate0, shape0, cu0), (r1, slow1, rate1, shape1, cu1) = res
    assert (r0, r1) == (0, 1)
    assert slow0 == slow1 == 137.5                   # every rank sees the slowest rank's time
    assert rate0 == rate1 == pytest.approx(2 * 1.0e12 * 10 / 0.1375)
    assert shape0 == shape1 and cu0 != cu1           # same shape, each replica its own documents


def test_single_process_needs_no_group():
    assert max_over_ranks(12.5) == 12.5
    assert whole_job_rate(1, 3.0, 4, 2000.0) == 6.0
    with pytest.raises(ValueError):
        whole_job_rate(1, 3.0, 0, 2000.0)


def test_rank_environment():
    e = rank_env({})
    assert (e.world, e.rank, e.local) == (1, 0, 0)
    e = rank_env({"WORLD_SIZE": "4", "RANK": "3", "LOCAL_RANK": "3"})
    assert (e.world, e.rank, e.local) == (4, 3, 3)
    with pytest.raises(ValueError):
        rank_env({"WORLD_SIZE": "2", "RANK": "2"})


def test_reference_arm_prints_from_rank_zero_only(monkeypatch, capsys):
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "bench_mod", os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = types.SimpleNamespace(workload="tiny", steps=1, warmup=3, gpus=2, noncausal=False)
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""
