"""bench.py's reference arm (the CPU oracle) on CPU: the JSON line it prints
carries the contract's keys, with the oracle as its own baseline and no
host-device traffic.  Budgets are shrunk so the test takes seconds."""

import argparse
import io
import json
import os
import sys
from contextlib import redirect_stdout

import pytest

pytest.importorskip("torch")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_the_contract_line(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    real = bench.oracle_rate
    monkeypatch.setattr(bench, "oracle_rate",
                        lambda wl, budget_s=0.0, seed=0, booked=None: real(wl, 0.05, seed, booked))
    args = argparse.Namespace(workload="nested_share", steps=2, warmup=3)
    out = io.StringIO()
    with redirect_stdout(out):
        bench.run_reference(args, 0, 1)
    lines = [ln for ln in out.getvalue().splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "nested_share"
    # the GPU arm prints the same config for the same workload
    from radix_tree_prefix_gb300 import workloads
    assert d["config"] == bench.config_of(workloads.nested_share(), 1)
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["cpu_baseline"]["host_cpus"] == os.cpu_count()
    assert d["cpu_baseline"]["blas_threads"] == 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_default_workload_is_the_largest_single_gpu_config():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.parse([]).workload == "multi_turn_chat"


def test_oracle_rate_counts_pairs_of_the_flow():
    """The oracle baseline's pair count equals the visible (query, key) pairs
    of the flow: extend query i sees i + 1 keys, decode step t sees the prompt
    and t + 1 decode tokens."""
    sys.path.insert(0, ROOT)
    import bench
    from radix_tree_prefix_gb300 import workloads
    wl = workloads.agent_loop(calls=3, preamble=20, lo=2, hi=5, decode_steps=2)
    trace, _ = bench.oracle_bookkeeping(wl)
    ext, dec = bench._pairs(trace, wl)
    want_e = sum(i + 1 for b in trace.batches for _, m, row in b for i in range(m, len(row)))
    want_d = sum(len(wl.prompt_tokens(r)) + t + 1 for w in wl.waves for r in w for t in range(2))
    assert (ext, dec) == (want_e, want_d)
    r = bench.oracle_rate(wl, budget_s=0.05, booked=(trace, 0.01))
    assert r["value"] > 0 and r["cores"] == 1 and "seeded requests" in r["sample"]


def test_other_ranks_print_nothing():
    sys.path.insert(0, ROOT)
    import bench

    out = io.StringIO()
    with redirect_stdout(out):
        bench.run_reference(argparse.Namespace(workload="nested_share", steps=1, warmup=3), 1, 2)
    assert out.getvalue() == ""
