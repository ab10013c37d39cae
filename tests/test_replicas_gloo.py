"""The N>1 path of bench.py on CPU: two replicas (gloo, world_size 2) each run
the request flow on their own cache, make identical cache decisions, and the
job's step time is the slowest rank's (max over ranks), its rate world x
units / that time.  The path has no data exchange between replicas, so the
only collectives are these reductions (and barriers)."""

import hashlib
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
dist = pytest.importorskip("torch.distributed")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import bench
    from radix_tree_prefix_gb300 import workloads
    from radix_tree_prefix_gb300.engine import Engine

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = workloads.nested_share()
        trace = Engine(wl, device=None).run()
        # each replica reports its own step time; the job takes the slowest
        my_seconds = 0.010 + 0.005 * rank
        seconds = bench.max_over_ranks(my_seconds, world, torch.device("cpu"))
        rate = bench.job_rate(trace.prefilled, seconds, world)
        dist.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            digest = hashlib.sha256(repr(trace.as_tuple()).encode()).hexdigest()
            f.write(f"{trace.prefilled} {digest} {seconds!r} {rate!r}\n")
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas_reduce_step_time(tmp_path):
    import torch.multiprocessing as mp

    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    rows = [open(tmp_path / f"rank{r}.txt").read().split() for r in range(world)]
    prefilled = {int(r[0]) for r in rows}
    traces = {r[1] for r in rows}
    seconds = {float(r[2]) for r in rows}
    rates = {float(r[3]) for r in rows}
    assert prefilled == {3060}          # the nested example's prefill count, on every rank
    assert len(traces) == 1             # identical cache decisions on both replicas
    assert seconds == {0.015}           # max over ranks, seen by every rank
    assert rates == {world * 3060 / 0.015}


def test_one_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.25, 1, torch.device("cpu")) == 0.25
    assert bench.job_rate(100, 0.5, 1) == 200.0
