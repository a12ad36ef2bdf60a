"""The multi-process path of bench.py on CPU (gloo, world size 2).

Rows are independent, so several GPUs run as replicas: every rank benches its
own batch and the job's value is all ranks' rows over the slowest rank's
time.  These tests run that host logic with two gloo ranks on the CPU: the
barrier, the max over ranks, the whole-job value and the per-rank inputs.
"""
import importlib.util
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench = _bench()
        dist.barrier()
        ms = bench.max_over_ranks(times[rank], dist, "cpu")
        value = bench.job_value(32, 100, world, ms)
        b = bench.make_workload("logits_chunk", rank)
        out_q.put((rank, ms, value, float(b["logits"][0, :8].float().sum())))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world, times = 2, [10.0, 12.5]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=300) for _ in range(world))
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [12.5, 12.5]                 # every rank holds the max
    assert res[0][2] == pytest.approx(32 * 100 * 2 / 0.0125)    # all ranks' rows / slowest time
    assert res[0][3] != res[1][3]                               # each rank streams its own batch


def test_one_process_is_unchanged():
    bench = _bench()
    assert bench.max_over_ranks(7.0, None, "cpu") == 7.0
    assert bench.job_value(32, 10, 1, 2.0) == pytest.approx(32 * 10 / 0.002)
