"""The N>1 path of bench.py on CPU: two replicas (gloo, world_size 2), each
with its own cache, run their subtree-affine share of the request flow
(fork_tree: one level-1 subtree per wave, waves round-robin over ranks) and
make exactly the oracle's decisions on that share; the shares are disjoint
and together cover the workload, so their prefilled tokens add up to the
one-replica run's; the job's step time is the slowest rank's and its rate the
units of all ranks over that time.  The path has no data exchange between
replicas: the only collectives are these reductions (and barriers)."""

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


def _small_fork_tree():
    from radix_tree_prefix_gb300 import workloads
    return workloads.fork_tree(branching=4, depth=3, level_tokens=20, decode_steps=3)


def _rank_main(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import bench
    from oracle.harness import run_bookkeeping
    from radix_tree_prefix_gb300 import workloads
    from radix_tree_prefix_gb300.engine import Engine

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = workloads.shard(_small_fork_tree(), rank, world)
        trace = Engine(wl, device=None).run()
        want, _ = run_bookkeeping(wl.oracle_waves(), wl.num_slots, wl.decode_steps)
        same = trace.as_tuple() == want.as_tuple()
        # each replica reports its own step time; the job takes the slowest
        my_seconds = 0.010 + 0.005 * rank
        seconds = bench.max_over_ranks(my_seconds, world, torch.device("cpu"))
        rate = bench.job_rate(trace.prefilled, seconds, world, torch.device("cpu"))
        dist.barrier()
        rids = sorted(r.rid for w in wl.waves for r in w)
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            digest = hashlib.sha256(repr(trace.as_tuple()).encode()).hexdigest()
            f.write(f"{trace.prefilled} {digest} {seconds!r} {rate!r} {int(same)} "
                    f"{','.join(map(str, rids))}\n")
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas_split_the_work(tmp_path):
    import torch.multiprocessing as mp

    sys.path.insert(0, ROOT)
    from radix_tree_prefix_gb300.engine import Engine

    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    rows = [open(tmp_path / f"rank{r}.txt").read().split() for r in range(world)]
    prefilled = [int(r[0]) for r in rows]
    assert all(r[4] == "1" for r in rows)               # each share bit-exact with the oracle
    assert rows[0][1] != rows[1][1]                       # different shares
    shares = [set(map(int, r[5].split(","))) for r in rows]
    full = _small_fork_tree()
    assert not (shares[0] & shares[1])                    # disjoint ...
    assert shares[0] | shares[1] == set(full.requests)    # ... and covering
    one = Engine(full, device=None).run()
    assert sum(prefilled) == one.prefilled                # subtrees share no prefix
    seconds = {float(r[2]) for r in rows}
    rates = {float(r[3]) for r in rows}
    assert seconds == {0.015}                             # max over ranks, seen by every rank
    assert rates == {sum(prefilled) / 0.015}              # all ranks' units / slowest time


def test_one_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.25, 1, torch.device("cpu")) == 0.25
    assert bench.job_rate(100, 0.5, 1) == 200.0


def test_shards_route_sessions_and_subtrees():
    """Chat sessions keep their replica from turn to turn; fork_tree waves
    (level-1 subtrees) go round-robin; one replica gets everything."""
    sys.path.insert(0, ROOT)
    from radix_tree_prefix_gb300 import workloads
    chat = workloads.multi_turn_chat(sessions=6, turns=3, system=10, user=5, decode_steps=2,
                                     layers=1)
    for rank in range(3):
        sh = workloads.shard(chat, rank, 3)
        sessions = {r.rid % 6 for w in sh.waves for r in w}
        assert sessions == {rank, rank + 3} and len(sh.waves) == 3
    ft = workloads.fork_tree(branching=3, depth=2, level_tokens=4, decode_steps=1)
    sh = workloads.shard(ft, 1, 2)
    assert [w[0].rid for w in sh.waves] == [ft.waves[1][0].rid]
    assert workloads.shard(ft, 0, 1) is ft
