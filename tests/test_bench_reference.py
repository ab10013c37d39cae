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
                        lambda wl, rows_of, budget_s=0.0, seed=0: real(wl, rows_of, 0.05, seed))
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
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_other_ranks_print_nothing():
    sys.path.insert(0, ROOT)
    import bench

    out = io.StringIO()
    with redirect_stdout(out):
        bench.run_reference(argparse.Namespace(workload="nested_share", steps=1, warmup=3), 1, 2)
    assert out.getvalue() == ""
